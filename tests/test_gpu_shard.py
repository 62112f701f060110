"""GPU parity of key-sharded decode ("Score a DSA sparse indexer in FP4", section "Decode context
parallelism"), through the C ABI: decode over key ranges against the oracle's range top-k, the
candidate merge against the oracle's merge, and the merge of every shard's list against the
unsharded decode call (bit for bit: same selected keys, same logits)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_sparse_attention_mxfp4_gb300 as fx
from fp4_sparse_attention_mxfp4_gb300 import shard
from gpu_helpers import DecodeRun, assert_topk_match, dev

pytestmark = pytest.mark.gpu


def _range_decode(run: DecodeRun, kb, ke):
    """The run's cache and queries scored over [kb[b], ke[b]) per sequence: (idx, val) [B, k]."""
    case = run.case
    sched = torch.zeros_like(run.sched)
    ws = torch.zeros_like(run.ws)
    idx = torch.full((case.batch, case.topk), -7, dtype=torch.int32, device="cuda")
    val = torch.full((case.batch, case.topk), 7.0, dtype=torch.float32, device="cuda")
    ke_d = dev(ke)
    fx.idx_fp4_build_decode_schedule_range(dev(kb), ke_d, run.max_batch, run.max_ctx, sched, status=run.status)
    fx.idx_fp4_decode_logits_topk(run.q_packed, run.q_scale, run.w, run.kv_p, run.kv_s, run.bt, ke_d, case.topk,
                                  sched, ws, idx, val, status=run.status)
    torch.cuda.synchronize()
    return idx, val


def _oracle_side(case):
    kv_p = np.full((case.layout.num_pages, 4, 64, 16), 0x77, np.uint8)
    kv_s = np.full((case.layout.num_pages, 4, 64), 0xFF, np.uint8)
    oracle.quant_and_cache(case.k_bf16, case.all_slots(), kv_p, kv_s)
    qp, qs = oracle.quantize_plain(case.q_bf16)
    return kv_p, kv_s, qp, qs


@pytest.mark.parametrize("lists,rows,k_in,topk", [(1, 3, 64, 64), (2, 16, 2048, 2048), (4, 5, 700, 1000),
                                                  (8, 2, 2048, 2048), (3, 4, 100, 512)])
def test_merge_candidates_matches_oracle(lists, rows, k_in, topk):
    rng = np.random.default_rng(lists * 100 + k_in)
    idx = np.stack([rng.permutation(1 << 20)[:lists * k_in].reshape(lists, k_in) for _ in range(rows)], axis=1)
    idx = idx.astype(np.int32)
    # fp32 values with many exact ties and a spread of magnitudes and signs; ~10% empty slots
    val = (rng.integers(-40, 40, size=idx.shape) * np.float32(0.37)).astype(np.float32)
    idx[rng.random(idx.shape) < 0.1] = -1
    out_i = torch.full((rows, topk), -7, dtype=torch.int32, device="cuda")
    out_v = torch.full((rows, topk), 7.0, dtype=torch.float32, device="cuda")
    fx.idx_fp4_merge_candidates(dev(val), dev(idx), topk, out_i, out_v)
    torch.cuda.synchronize()
    ei, ev = oracle.merge_candidates(val.astype(np.float64), idx, topk)
    gi, gv = out_i.cpu().numpy(), out_v.cpu().numpy()
    for r in range(rows):
        n = int((ei[r] >= 0).sum())
        order = np.argsort(ei[r, :n])
        assert np.array_equal(gi[r, :n], ei[r, :n][order]), f"row {r}: selected keys differ"
        assert np.array_equal(gv[r, :n].astype(np.float64), ev[r, :n][order]), f"row {r}: values differ"
        assert np.all(gi[r, n:] == -1) and np.all(np.isneginf(gv[r, n:]))


def test_range_decode_matches_oracle():
    case = synth.decode_case("range", 23, [40000, 5000, 300, 131072], 64, 2048)
    run = DecodeRun(case, debug_logits=False)
    kb = np.array([1024, 0, 128, 65536], np.int32)
    ke = np.array([39999, 4097, 300, 100000], np.int32)
    idx, val = _range_decode(run, kb, ke)
    assert int(run.status.item()) == 0
    kv_p, kv_s, qp, qs = _oracle_side(case)
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    for b in range(case.batch):
        lg = oracle.row_logits(qp, qs, case.w, b, kv_p, kv_s, case.layout.block_tables[b], int(kb[b]), int(ke[b]))
        sel = gi[b][gi[b] >= 0]
        assert np.all((sel >= kb[b]) & (sel < ke[b]))
        rel_i = np.where(gi[b] >= 0, gi[b] - kb[b], -1).astype(np.int32)
        assert_topk_match(rel_i, gv[b], lg, case.topk, f"seq {b} range")


@pytest.mark.parametrize("world", [2, 3, 8])
def test_sharded_decode_equals_unsharded(world):
    ctx = [200000, 3, 150001, 64, 99999, 131072]
    case = synth.decode_case(f"shards{world}", 29, ctx, 64, 2048)
    run = DecodeRun(case, debug_logits=False).run()
    assert int(run.status.item()) == 0
    parts = [_range_decode(run, kb, ke) for kb, ke in shard.shard_ranges(case.ctx_lens, world)]
    assert int(run.status.item()) == 0
    cand_i = torch.stack([p[0] for p in parts])
    cand_v = torch.stack([p[1] for p in parts])
    out_i = torch.empty_like(run.topk_idx)
    out_v = torch.empty_like(run.topk_val)
    fx.idx_fp4_merge_candidates(cand_v, cand_i, case.topk, out_i, out_v)
    torch.cuda.synchronize()
    assert torch.equal(out_i, run.topk_idx)
    assert torch.equal(out_v.view(torch.int32), run.topk_val.view(torch.int32))

