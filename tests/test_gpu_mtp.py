"""GPU parity of decode with next_n verify rows per sequence (speculative decoding), against the
oracle, through the C ABI.

The rows are expressed through the prefill call: sequence b is a request of next_n rows sharing
its page table, and row j sees keys [0, ctx_b - next_n + 1 + j), so the last key of the step is
visible to the last row only. Long contexts are scored in key chunks whose candidate lists are
merged.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_sparse_attention_mxfp4_gb300 as fx
from gpu_helpers import assert_cache_equal, assert_logits_close, assert_topk_match, bf16_dev, dev, new_cache, oracle_cache

pytestmark = pytest.mark.gpu


def _run(case: synth.MtpCase):
    B, H, R = case.batch, case.heads, case.batch * case.next_n
    kv_p, kv_s = new_cache(case.layout.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qp = torch.empty((R, H, 64), dtype=torch.uint8, device="cuda")
    qs = torch.empty((R, H, 4), dtype=torch.uint8, device="cuda")
    fx.idx_fp4_quant_and_cache(bf16_dev(case.k_bf16), dev(case.all_slots()), kv_p, kv_s, q_bf16=bf16_dev(case.q_bf16),
                               q_packed=qp, q_scale=qs, status=status)
    max_ctx = int(case.ctx_lens.max())
    ws = torch.zeros(fx.idx_fp4_prefill_workspace_bytes(B, R, H, max_ctx, case.topk), dtype=torch.uint8,
                     device="cuda")
    idx = torch.full((R, case.topk), -7, dtype=torch.int32, device="cuda")
    val = torch.full((R, case.topk), 7.0, dtype=torch.float32, device="cuda")
    lg = torch.full((R, max_ctx), float("nan"), dtype=torch.float32, device="cuda")
    fx.idx_fp4_prefill_logits_topk(qp, qs, dev(case.w), kv_p, kv_s, dev(case.layout.block_tables), dev(case.ctx_lens),
                                   dev(case.cu_seqlens()), dev(case.row_ends()), case.topk, max_ctx, ws, idx, val,
                                   logits_debug=lg, status=status)
    torch.cuda.synchronize()
    return kv_p, kv_s, qp, qs, idx.cpu().numpy(), val.cpu().numpy(), lg.cpu().numpy(), int(status.item())


def _check(case, out, rows):
    kv_p, kv_s, qp, qs, idx, val, lg, status = out
    ref_p, ref_s = oracle_cache(case.layout.num_pages, case.k_bf16, case.all_slots())
    assert_cache_equal(kv_p, kv_s, ref_p, ref_s)
    rqp, rqs = oracle.quantize_plain(case.q_bf16)
    assert np.array_equal(qp.cpu().numpy(), rqp) and np.array_equal(qs.cpu().numpy(), rqs)
    ends = case.row_ends()
    for r in rows:
        b, e = r // case.next_n, int(ends[r])
        ref = oracle.row_logits(rqp, rqs, case.w, r, ref_p, ref_s, case.layout.block_tables[b], 0, e)
        assert_logits_close(lg[r, :e], ref, f"{case.name} row {r}")
        assert np.all(np.isnan(lg[r, e:])), f"{case.name} row {r} wrote logits past its last key"
        assert_topk_match(idx[r], val[r], ref, case.topk, f"{case.name} row {r}")
    assert status == 0, f"status {status:#x}"


@pytest.mark.parametrize("heads,next_n,topk", [(64, 2, 2048), (32, 3, 64), (128, 2, 512)])
def test_mtp_verify_rows(heads, next_n, topk):
    # short and long contexts, one exactly next_n keys long, one past a key chunk of the scorer
    case = synth.mtp_case(f"mtp_h{heads}_n{next_n}", 70 + next_n, [300, next_n, 5000, 40000], heads, topk, next_n)
    out = _run(case)
    _check(case, out, range(case.batch * case.next_n))


def test_mtp_full_size_sampled():
    """The 16 x 131072 workload with two verify rows per sequence: every row of two sequences."""
    case = synth.mtp_config()
    out = _run(case)
    n = case.next_n
    _check(case, out, [0, 1, (case.batch - 1) * n, (case.batch - 1) * n + 1])


def _run_decode(case: synth.MtpCase, logits=True):
    """The same rows through the decode-shaped call: one pass over each sequence's keys for all
    next_n rows (next_n * heads <= 128)."""
    B, H, R, n = case.batch, case.heads, case.batch * case.next_n, case.next_n
    kv_p, kv_s = new_cache(case.layout.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qp = torch.empty((R, H, 64), dtype=torch.uint8, device="cuda")
    qs = torch.empty((R, H, 4), dtype=torch.uint8, device="cuda")
    fx.idx_fp4_quant_and_cache(bf16_dev(case.k_bf16), dev(case.all_slots()), kv_p, kv_s, q_bf16=bf16_dev(case.q_bf16),
                               q_packed=qp, q_scale=qs, status=status)
    max_ctx = int(case.ctx_lens.max())
    ctx = dev(case.ctx_lens)
    sched = torch.zeros(fx.idx_fp4_decode_schedule_bytes(B, max_ctx), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(fx.idx_fp4_decode_mtp_workspace_bytes(B, max_ctx, case.topk, n), dtype=torch.uint8,
                     device="cuda")
    idx = torch.full((R, case.topk), -7, dtype=torch.int32, device="cuda")
    val = torch.full((R, case.topk), 7.0, dtype=torch.float32, device="cuda")
    lg = torch.full((R, max_ctx), float("nan"), dtype=torch.float32, device="cuda") if logits else None
    fx.idx_fp4_build_decode_schedule_mtp(ctx, n, B, max_ctx, sched, status=status)
    fx.idx_fp4_decode_mtp_logits_topk(qp, qs, dev(case.w), kv_p, kv_s, dev(case.layout.block_tables), ctx, n,
                                      case.topk, sched, ws, idx, val, logits_debug=lg, status=status)
    torch.cuda.synchronize()
    lg_np = lg.cpu().numpy() if logits else None
    return (kv_p, kv_s, qp, qs, idx.cpu().numpy(), val.cpu().numpy(), lg_np, int(status.item())), sched


@pytest.mark.parametrize("heads,next_n,topk", [(64, 2, 2048), (32, 2, 64), (16, 2, 512), (32, 4, 64),
                                               (16, 4, 2048)])
def test_decode_mtp_rows(heads, next_n, topk):
    # contexts: one exactly next_n keys long, ragged tile tails, one shorter than k for some rows,
    # and sequences that span several CTAs of the decode grid
    ctx = [300, next_n, 5000, 40000, 129, 2049, 200000]
    case = synth.mtp_case(f"dmtp_h{heads}_n{next_n}_k{topk}", 80 + next_n + heads, ctx, heads, topk, next_n)
    out, _ = _run_decode(case)
    _check(case, out, range(case.batch * case.next_n))


def test_decode_mtp_matches_prefill_form():
    """The decode-shaped call and the prefill call select the same keys for the same verify rows."""
    case = synth.mtp_case("dmtp_vs_prefill", 91, [7000, 33000, 2], 64, 2048, 2)
    a, _ = _run_decode(case)
    b = _run(case)
    assert np.array_equal(a[4], b[4])
    assert np.array_equal(a[5].view(np.int32), b[5].view(np.int32))


def test_decode_mtp_full_size_sampled():
    """16 x 131072 keys with two verify rows per sequence through the decode-shaped call: every
    row of two sequences."""
    case = synth.mtp_config()
    out, _ = _run_decode(case)
    n = case.next_n
    _check(case, out, [0, 1, (case.batch - 1) * n, (case.batch - 1) * n + 1])


def test_decode_mtp_several_rounds():
    """More keys than one pass of the grid holds at next_n 4 (a range is at most 8192 keys), so
    the sequences' segments from different rounds are merged: rows of the first and last
    sequences against the oracle."""
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 256)
    per_round = sms * 64 * 128
    nseq = 8
    L = -(-(per_round * 5 // 4) // nseq) + 1
    case = synth.mtp_case("dmtp_rounds", 95, [L] * (nseq - 1) + [L - 333], 32, 2048, 4)
    out, sched = _run_decode(case, logits=False)
    hdr = sched[:64].cpu().numpy().view(np.int32)
    assert hdr[5] >= 2, f"expected several rounds, header {hdr[:16]}"
    kv_p, kv_s, qp, qs, idx, val, _, status = out
    assert status == 0, f"status {status:#x}"
    rqp, rqs = oracle.quantize_plain(case.q_bf16)
    ref_p, ref_s = oracle_cache(case.layout.num_pages, case.k_bf16, case.all_slots())
    ends = case.row_ends()
    for r in [0, 3, (nseq - 1) * 4, (nseq - 1) * 4 + 3]:
        b, e = r // 4, int(ends[r])
        ref = oracle.row_logits(rqp, rqs, case.w, r, ref_p, ref_s, case.layout.block_tables[b], 0, e)
        assert_topk_match(idx[r], val[r], ref, case.topk, f"row {r}")
