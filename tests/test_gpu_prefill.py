"""GPU parity of the causal prefill scorer against the oracle, through the C ABI.

Each prefill step writes its tokens' keys into the cache (the writer) and then scores every row
of the step against keys [0, row_end) of its request. Padding rows (row_end 0, folded into the
step's last request) must come out as all -1 and read nothing: unwritten cache rows hold the
NaN scale sentinel, so any stray read would poison a logit.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_sparse_attention_mxfp4_gb300 as fx
from gpu_helpers import (assert_cache_equal, assert_logits_close, assert_topk_match, bf16_dev, dev, new_cache,
                         oracle_cache)

pytestmark = pytest.mark.gpu


class PrefillRun:
    def __init__(self, case: synth.PrefillCase, debug_logits=True):
        self.case = case
        self.kv_p, self.kv_s = new_cache(case.layout.num_pages)
        self.bt_all = case.layout.block_tables
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.debug = debug_logits
        self.slots_all = case.token_slots()

    def step(self, st: synth.PrefillStep):
        case, H = self.case, self.case.heads
        R = st.rows
        toks = st.token_ids
        # this step's keys go into the cache first
        fx.idx_fp4_quant_and_cache(bf16_dev(case.k_bf16[toks]), dev(self.slots_all[toks]), self.kv_p, self.kv_s,
                                   status=self.status)
        # queries of the step; padding rows get zero weights and zero queries
        q = np.zeros((R, H, 128), np.uint16)
        q[:st.real_rows] = case.q_bf16[toks]
        w = np.zeros((R, H), np.float32)
        w[:st.real_rows] = case.w[toks]
        qp = torch.empty((R, H, 64), dtype=torch.uint8, device="cuda")
        qs = torch.empty((R, H, 4), dtype=torch.uint8, device="cuda")
        fx.idx_fp4_quant_and_cache(bf16_dev(case.k_bf16[:0]), dev(np.zeros(0, np.int32)), self.kv_p, self.kv_s,
                                   q_bf16=bf16_dev(q), q_packed=qp, q_scale=qs)
        bt = dev(self.bt_all[st.requests])
        max_ctx = max(int(st.ctx_lens.max()), 1)
        ws = torch.zeros(fx.idx_fp4_prefill_workspace_bytes(len(st.requests), R, H, max_ctx, case.topk),
                         dtype=torch.uint8, device="cuda")
        idx = torch.full((R, case.topk), -7, dtype=torch.int32, device="cuda")
        val = torch.full((R, case.topk), 7.0, dtype=torch.float32, device="cuda")
        width = max(int(st.row_ends.max()), 1)
        lg = torch.full((R, width), float("nan"), dtype=torch.float32, device="cuda") if self.debug else None
        fx.idx_fp4_prefill_logits_topk(qp, qs, dev(w), self.kv_p, self.kv_s, bt, dev(st.ctx_lens), dev(st.cu_seqlens),
                                       dev(st.row_ends), case.topk, max_ctx, ws, idx, val, logits_debug=lg,
                                       status=self.status)
        torch.cuda.synchronize()
        return q, w, qp, qs, idx.cpu().numpy(), val.cpu().numpy(), (lg.cpu().numpy() if lg is not None else None)


def _check_step(run, st, out, kv_ref, rows):
    case = run.case
    q, w, qp, qs, idx, val, lg = out
    rqp, rqs = oracle.quantize_plain(q)
    assert np.array_equal(qp.cpu().numpy(), rqp) and np.array_equal(qs.cpu().numpy(), rqs)
    kv_p, kv_s = kv_ref
    group = np.searchsorted(st.cu_seqlens, np.arange(st.rows), side="right") - 1
    for r in rows:
        g = group[r]
        e = int(st.row_ends[r])
        table = run.bt_all[st.requests[g]]
        ref = oracle.row_logits(rqp, rqs, w, r, kv_p, kv_s, table, 0, e)
        if lg is not None and e > 0:
            assert_logits_close(lg[r, :e], ref, f"{case.name} row {r}")
        assert_topk_match(idx[r], val[r], ref, case.topk, f"{case.name} row {r}")
        if e == 0:
            assert lg is None or np.all(np.isnan(lg[r])), "a padding row wrote logits"


def _run_case(case, rows_per_step=None, seed=0):
    run = PrefillRun(case)
    ref_p = np.full((case.layout.num_pages, 4, 64, 16), 0x77, np.uint8)
    ref_s = np.full((case.layout.num_pages, 4, 64), 0xFF, np.uint8)
    rng = synth.Rng(seed)
    for si, st in enumerate(case.steps):
        out = run.step(st)
        oracle.quant_and_cache(case.k_bf16[st.token_ids], run.slots_all[st.token_ids], ref_p, ref_s)
        if si == 0 or si == len(case.steps) - 1:
            assert_cache_equal(run.kv_p, run.kv_s, ref_p, ref_s)
        if rows_per_step is None:
            rows = range(st.rows)
        else:
            pick = set(rng.integers(0, st.rows - 1, rows_per_step).tolist())
            pick |= {0, st.real_rows - 1, st.rows - 1}
            pick |= set(st.cu_seqlens[:-1].tolist())
            rows = sorted(r for r in pick if r < st.rows)
        _check_step(run, st, out, (ref_p, ref_s), rows)
    assert int(run.status.item()) == 0, f"status {int(run.status.item()):#x}"


def test_prefill_small_full_check():
    # three short requests, steps of 61 real rows padded to a multiple of 8, topk larger and
    # smaller than the rows' key counts
    case = synth.prefill_case("small", 41, [150, 70, 201], 64, 96, budget=64, real_per_step=61, pad_to=8)
    _run_case(case)


@pytest.mark.parametrize("heads", [16, 32, 128])
def test_prefill_heads(heads):
    case = synth.prefill_case(f"heads{heads}", 42 + heads, [130, 67], heads, 64, budget=128, real_per_step=125,
                              pad_to=8)
    _run_case(case)


def test_prefill_workload_pad8_sampled():
    """Four prompts of 2634..4295 tokens, 512-row steps with padding rows, topk 2048."""
    _run_case(synth.prefill_config("pad8"), rows_per_step=12, seed=5)


def test_prefill_workload_odd_total_sampled():
    """The same prompts with steps whose padded row count stays a non-multiple of 8."""
    _run_case(synth.prefill_config("odd"), rows_per_step=6, seed=6)


def test_prefill_identity_table_small_full_check():
    # two requests staged back to back in a flat pool: each request's page table is consecutive pages
    case = synth.prefill_case("flat_small", 45, [150, 201], 64, 96, budget=64, real_per_step=61, pad_to=8,
                              contiguous=True)
    assert np.array_equal(case.layout.block_tables[1, :4], np.arange(3, 7))
    _run_case(case)


def test_prefill_identity_table_long_prompt_sampled():
    """One 16384-token prompt over an identity page table: rows past 8192 keys are scored in key
    chunks whose candidate lists are merged."""
    case = synth.prefill_flat_config()
    assert np.array_equal(case.layout.block_tables[0], np.arange(case.layout.num_pages))
    _run_case(case, rows_per_step=4, seed=7)


def test_prefill_bad_rows_flagged():
    case = synth.prefill_case("bad", 43, [100], 16, 32, budget=104, real_per_step=100, pad_to=8)
    run = PrefillRun(case)
    st = case.steps[0]
    st.row_ends = st.row_ends.copy()
    st.row_ends[3] = 5000  # past the request's context: clamped and flagged
    run.step(st)
    assert int(run.status.item()) & fx.DEV_BAD_ROWS
