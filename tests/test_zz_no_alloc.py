"""The decode entry point that allocates nothing, against the regular one.

idx_fp4_decode_logits_topk_static serves callers that cannot allocate device memory (for
example code running inside an allocator or memory-pool hook, or a runtime that owns every
device allocation): instead of a caller workspace it keeps the candidate lists of split
sequences in a fixed array the library holds on each GPU. Its results must match the regular
call's. Two calls in a row, with different shapes, check that the second is not disturbed by
what the first left in the shared array. This file is collected last on purpose.
"""
import pytest
import torch

import synth
import fp4_sparse_attention_mxfp4_gb300 as fx
from gpu_helpers import DecodeRun

pytestmark = pytest.mark.gpu


def _regular(case):
    run = DecodeRun(case, debug_logits=False)
    run.run()
    return run, run.topk_idx.clone(), run.topk_val.clone()


def _static(run):
    idx = torch.full_like(run.topk_idx, -7)
    val = torch.full_like(run.topk_val, 7.0)
    fx.idx_fp4_decode_logits_topk_static(run.q_packed, run.q_scale, run.w, run.kv_p, run.kv_s, run.bt, run.ctx,
                                         run.case.topk, run.max_ctx, run.sched, idx, val, status=run.status)
    torch.cuda.synchronize()
    return idx, val


def _compare(ref_idx, ref_val, idx, val, what):
    # The static call is the regular decode call with another scratch area: same schedule, same
    # kernels, deterministic passes. Its outputs must equal the regular call's bit for bit, which
    # also shows that nothing left in the shared array by an earlier call leaks into a later one.
    assert torch.equal(ref_idx, idx), f"{what}: {int((ref_idx != idx).sum())} indices differ"
    assert torch.equal(ref_val.view(torch.int32), val.view(torch.int32)), f"{what}: values differ bitwise"


def test_static_scratch_matches_workspace_call_twice():
    # sequences long enough to be split over many CTAs, so the candidate lists are used
    case_a = synth.decode_case("static_a", 51, [40000, 23000, 3000], 64, 512)
    case_b = synth.decode_case("static_b", 52, [30000, 50000], 32, 1024)
    run_a, ref_ia, ref_va = _regular(case_a)
    run_b, ref_ib, ref_vb = _regular(case_b)
    assert int(run_a.status.item()) == 0 and int(run_b.status.item()) == 0
    ia, va = _static(run_a)
    ib, vb = _static(run_b)  # right after the first call: reuses what it left in the array
    _compare(ref_ia, ref_va, ia, va, "first call")
    _compare(ref_ib, ref_vb, ib, vb, "second call")
    assert int(run_a.status.item()) == 0 and int(run_b.status.item()) == 0


def test_static_scratch_rejects_batches_beyond_its_size():
    need = fx.idx_fp4_decode_static_bytes(64, 1 << 20, 2048)
    assert need > fx.STATIC_SCRATCH_BYTES
    # the C entry point refuses before touching any pointer or launching anything
    code = fx.lib().idx_fp4_decode_logits_topk_static(None, None, None, None, None, 1, None, 1, None, 64, 64, 2048,
                                                      1 << 20, None, 0, None, None, None, 0, None, None)
    assert code == 3  # IDX_FP4_ERR_CAPACITY
