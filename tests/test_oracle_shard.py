"""Key-sharded decode on CPU ("Score a DSA sparse indexer in FP4", section "Decode context
parallelism"): the oracle's range top-k and candidate merge pinned against numpy brute force,
the shard bookkeeping, and a world-size-2 gloo run in which each rank scores its own key range
with the oracle, the ranks all-gather their lists and the merge equals the unsharded decode."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import synth
from fp4_sparse_attention_mxfp4_gb300 import shard


def _brute_topk(vals, idx, k):
    """numpy: the k best (value desc, index asc) of (vals, idx) pairs."""
    order = np.lexsort((idx, -vals))[:k]
    return idx[order], vals[order]


def test_merge_matches_brute_force_with_ties_and_empties():
    rng = np.random.default_rng(5)
    for lists, rows, k_in, k in [(1, 3, 8, 5), (3, 4, 16, 20), (8, 2, 64, 64), (2, 5, 7, 30)]:
        # values from a small set (many exact ties), distinct indices per row, ~20% empty slots
        idx = np.stack([rng.permutation(10000)[:lists * k_in].reshape(lists, k_in) for _ in range(rows)], axis=1)
        idx = idx.astype(np.int32)
        vals = rng.integers(-3, 4, size=idx.shape).astype(np.float64) * 0.5
        idx[rng.random(idx.shape) < 0.2] = -1
        got_i, got_v = oracle.merge_candidates(vals, idx, k)
        for r in range(rows):
            ok = idx[:, r, :] >= 0
            ei, ev = _brute_topk(vals[:, r, :][ok], idx[:, r, :][ok], k)
            n = len(ei)
            assert np.array_equal(got_i[r, :n], ei) and np.array_equal(got_v[r, :n], ev)
            assert np.all(got_i[r, n:] == -1) and np.all(np.isneginf(got_v[r, n:]))


def _tiny_decode():
    case = synth.decode_case("shard_tiny", 17, [700, 129, 1, 0, 385], 16, 40)
    kv_p = np.full((case.layout.num_pages, 4, 64, 16), 0x77, np.uint8)
    kv_s = np.full((case.layout.num_pages, 4, 64), 0xFF, np.uint8)
    oracle.quant_and_cache(case.k_bf16, case.all_slots(), kv_p, kv_s)
    qp, qs = oracle.quantize_plain(case.q_bf16)
    return case, kv_p, kv_s, qp, qs


def test_range_topk_matches_brute_force():
    case, kv_p, kv_s, qp, qs = _tiny_decode()
    kb = np.array([128, 0, 0, 0, 256], np.int32)
    ke = np.array([600, 129, 1, 0, 385], np.int32)
    got_i, got_v = oracle.range_topk(qp, qs, case.w, kv_p, kv_s, case.layout.block_tables, kb, ke, case.topk)
    for b in range(case.batch):
        lg = oracle.row_logits(qp, qs, case.w, b, kv_p, kv_s, case.layout.block_tables[b], int(kb[b]), int(ke[b]))
        ei, ev = _brute_topk(lg, np.arange(kb[b], ke[b], dtype=np.int32), case.topk)
        n = len(ei)
        assert np.array_equal(got_i[b, :n], ei) and np.array_equal(got_v[b, :n], ev)
        assert np.all(got_i[b, n:] == -1)


def test_shard_ranges_partition_each_sequence():
    ctx = np.array([0, 1, 127, 128, 129, 1000, 131072, 5], np.int32)
    for world in (1, 2, 3, 4, 8):
        r = shard.shard_ranges(ctx, world)
        assert len(r) == world
        assert np.array_equal(r[0][0], np.zeros_like(ctx)) and np.array_equal(r[-1][1], ctx)
        for w in range(world):
            kb, ke = r[w]
            assert np.all(kb % shard.TILE == 0) and np.all(kb <= ke) and np.all(ke <= ctx)
            if w:
                assert np.array_equal(kb, r[w - 1][1])


def test_merged_shards_equal_unsharded_decode():
    case, kv_p, kv_s, qp, qs = _tiny_decode()
    full_i, full_v, _ = oracle.decode_topk(qp, qs, case.w, kv_p, kv_s, case.layout.block_tables, case.ctx_lens,
                                           case.topk)
    for world in (2, 3, 5):
        parts = [oracle.range_topk(qp, qs, case.w, kv_p, kv_s, case.layout.block_tables, kb, ke, case.topk)
                 for kb, ke in shard.shard_ranges(case.ctx_lens, world)]
        mi, mv = oracle.merge_candidates(np.stack([p[1] for p in parts]), np.stack([p[0] for p in parts]), case.topk)
        assert np.array_equal(mi, full_i) and np.array_equal(mv, full_v)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case, kv_p, kv_s, qp, qs = _tiny_decode()
    kb, ke = shard.shard_ranges(case.ctx_lens, world)[rank]
    li, lv = oracle.range_topk(qp, qs, case.w, kv_p, kv_s, case.layout.block_tables, kb, ke, case.topk)
    gi, gv = shard.gather_candidates(torch.from_numpy(li), torch.from_numpy(lv))
    mi, mv = oracle.merge_candidates(gv.numpy(), gi.numpy(), case.topk)
    full_i, full_v, _ = oracle.decode_topk(qp, qs, case.w, kv_p, kv_s, case.layout.block_tables, case.ctx_lens,
                                           case.topk)
    out[rank] = bool(np.array_equal(mi, full_i) and np.array_equal(mv, full_v))
    dist.destroy_process_group()


def test_sharded_decode_world2_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert out[0] and out[1]
