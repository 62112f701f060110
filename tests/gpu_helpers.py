"""Shared pieces of the GPU parity tests: device setup through the C ABI and the comparisons.

The CUDA path and the oracle each quantise the same seeded bf16 inputs on their own; the
tests compare the bytes both produced, then each side scores its own cache.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import fp4_sparse_attention_mxfp4_gb300 as fx

TOL = 1e-4  # |gpu - ref| <= TOL * (1 + |ref|)
PACKED_SENTINEL = 0x77
SCALE_SENTINEL = 0xFF  # e8m0 NaN: any read of an unwritten row poisons its logit


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def new_cache(num_pages: int):
    kv_p = torch.full((num_pages, 4, 64, 16), PACKED_SENTINEL, dtype=torch.uint8, device="cuda")
    kv_s = torch.full((num_pages, 4, 64), SCALE_SENTINEL, dtype=torch.uint8, device="cuda")
    return kv_p, kv_s


def oracle_cache(num_pages: int, k_bf16, slots):
    kv_p = np.full((num_pages, 4, 64, 16), PACKED_SENTINEL, np.uint8)
    kv_s = np.full((num_pages, 4, 64), SCALE_SENTINEL, np.uint8)
    n = oracle.quant_and_cache(k_bf16, slots, kv_p, kv_s)
    assert n == int((np.asarray(slots) >= 0).sum())
    return kv_p, kv_s


def bf16_dev(bits):
    return dev(bits.view(np.int16))


class DecodeRun:
    """Writer + schedule + decode scorer for one DecodeCase, all through the C ABI."""

    def __init__(self, case: synth.DecodeCase, max_batch=None, max_ctx=None, debug_logits=True):
        self.case = case
        B, H = case.batch, case.heads
        self.kv_p, self.kv_s = new_cache(case.layout.num_pages)
        self.q_packed = torch.empty((B, H, 64), dtype=torch.uint8, device="cuda")
        self.q_scale = torch.empty((B, H, 4), dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        slots = case.all_slots()
        fx.idx_fp4_quant_and_cache(bf16_dev(case.k_bf16), dev(slots), self.kv_p, self.kv_s,
                                   q_bf16=bf16_dev(case.q_bf16), q_packed=self.q_packed, q_scale=self.q_scale,
                                   status=self.status)
        self.w = dev(case.w)
        self.bt = dev(case.layout.block_tables)
        self.ctx = dev(case.ctx_lens)
        self.max_batch = max_batch or B
        self.max_ctx = max_ctx or int(case.ctx_lens.max())
        self.sched = torch.zeros(fx.idx_fp4_decode_schedule_bytes(self.max_batch, self.max_ctx), dtype=torch.uint8,
                                 device="cuda")
        self.ws = torch.zeros(fx.idx_fp4_decode_workspace_bytes(self.max_batch, self.max_ctx, case.topk),
                              dtype=torch.uint8, device="cuda")
        self.topk_idx = torch.full((B, case.topk), -7, dtype=torch.int32, device="cuda")
        self.topk_val = torch.full((B, case.topk), 7.0, dtype=torch.float32, device="cuda")
        self.logits = None
        if debug_logits:
            self.logits = torch.full((B, max(self.max_ctx, 1)), float("nan"), dtype=torch.float32, device="cuda")

    def schedule(self):
        fx.idx_fp4_build_decode_schedule(self.ctx, self.max_batch, self.max_ctx, self.sched, status=self.status)

    def score(self):
        fx.idx_fp4_decode_logits_topk(self.q_packed, self.q_scale, self.w, self.kv_p, self.kv_s, self.bt, self.ctx,
                                      self.case.topk, self.sched, self.ws, self.topk_idx, self.topk_val,
                                      logits_debug=self.logits, status=self.status)

    def run(self):
        self.schedule()
        self.score()
        torch.cuda.synchronize()
        return self


def assert_cache_equal(kv_p_gpu, kv_s_gpu, kv_p_ref, kv_s_ref):
    gp, gs = kv_p_gpu.cpu().numpy(), kv_s_gpu.cpu().numpy()
    bad_p = np.flatnonzero(gp.reshape(-1) != kv_p_ref.reshape(-1))
    bad_s = np.flatnonzero(gs.reshape(-1) != kv_s_ref.reshape(-1))
    assert bad_p.size == 0, f"{bad_p.size} packed bytes differ, first at {bad_p[:5]}"
    assert bad_s.size == 0, f"{bad_s.size} scale bytes differ, first at {bad_s[:5]}"


def assert_logits_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(ref)), f"{what}: oracle logits not finite"
    err = np.abs(gpu - ref)
    lim = TOL * (1.0 + np.abs(ref))
    bad = np.flatnonzero(~(err <= lim))
    assert bad.size == 0, (f"{what}: {bad.size}/{ref.size} logits off, worst at {bad[np.argmax(err[bad])]}: "
                           f"gpu {gpu[bad[0]]} ref {ref[bad[0]]}")


def assert_topk_match(idx_row, val_row, ref_logits, k, what=""):
    """The GPU's top-k set equals the oracle's up to ties within tolerance; values match; the
    indices come in ascending order followed by -1 padding (value -inf)."""
    idx_row = np.asarray(idx_row)
    n_keys = ref_logits.shape[0]
    n = min(k, n_keys)
    sel = idx_row[:n]
    assert np.all(idx_row[n:] == -1), f"{what}: padding not -1"
    assert np.all(sel >= 0) and np.all(sel < n_keys), f"{what}: index out of range"
    assert np.all(np.diff(sel) > 0), f"{what}: indices not strictly ascending"
    if val_row is not None:
        val_row = np.asarray(val_row, np.float64)
        assert np.all(np.isneginf(val_row[n:])), f"{what}: padding values not -inf"
        assert_logits_close(val_row[:n], ref_logits[sel], what + " values")
    if n == 0:
        return
    order = np.lexsort((np.arange(n_keys), -ref_logits))[:n]
    vk = ref_logits[order[-1]]
    diff = np.setxor1d(sel, order)
    if diff.size:
        off = np.abs(ref_logits[diff] - vk)
        assert np.all(off <= TOL * (1 + abs(vk))), (
            f"{what}: {diff.size} keys differ beyond ties, worst gap {off.max()} at threshold {vk}")
