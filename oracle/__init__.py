"""Test oracle for the MXFP4 DSA lightning indexer (fp64, CPU, plain C++).

THIS IS TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import it. The product library
never imports, links or executes anything here, and this package imports
nothing from the product package.

The arithmetic lives in ``oracle.cpp`` (see its header for the passages each
function restates); this module compiles it with g++ and wraps it with ctypes
and numpy. Nothing here computes any part of the method itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

HEAD_DIM = 128
PAGE = 64


def build(force: bool = False) -> str:
    """Compile oracle.cpp into oracle/_build/liboracle.so (portable flags only)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            sig = {
                "orc_version": (i32, []),
                "orc_scale_slot": (i32, [i32]),
                "orc_block_exponent": (i32, [dbl]),
                "orc_e2m1_round": (i32, [dbl]),
                "orc_e2m1_value": (dbl, [i32]),
                "orc_quantize_plain": (None, [P, i64, P, P]),
                "orc_dequantize_plain": (None, [P, P, i64, P]),
                "orc_quant_and_cache": (i64, [P, i64, P, P, P, i64]),
                "orc_read_key": (None, [P, P, i64, i32, P]),
                "orc_decode_logits": (None, [P, P, P, P, P, P, i64, P, i32, i32, P, i64, i32]),
                "orc_row_logits": (None, [P, P, P, i64, i32, P, P, P, i64, i64, P]),
                "orc_prefill_logits": (None, [P, P, P, P, P, P, i64, P, P, i32, i32, i32, P, i64, i32]),
                "orc_select_topk": (None, [P, i64, i32, P, P]),
                "orc_decode_topk": (None, [P, P, P, P, P, P, i64, P, i32, i32, i32, P, i64, P, P, i32]),
                "orc_prefill_topk": (None, [P, P, P, P, P, P, i64, P, P, i32, i32, i32, i32, P, i64, P, P, i32]),
                "orc_range_topk": (None, [P, P, P, P, P, P, i64, P, P, i32, i32, i32, P, i64, P, P, i32]),
                "orc_merge_candidates": (None, [P, P, i32, i32, i32, i32, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar helpers ------------------------------------------------------------------

def scale_slot(row: int) -> int:
    return _load().orc_scale_slot(int(row))


def block_exponent(amax: float) -> int:
    return _load().orc_block_exponent(float(amax))


def e2m1_round(y: float) -> int:
    return _load().orc_e2m1_round(float(y))


def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


# ---- quantiser and cache -------------------------------------------------------------

def quantize_plain(x_bf16: np.ndarray):
    """bf16 bit patterns [..., 128] (uint16) -> (packed uint8 [..., 64], scales uint8 [..., 4])."""
    x = _c(x_bf16, np.uint16)
    lead = x.shape[:-1]
    assert x.shape[-1] == HEAD_DIM
    n = int(np.prod(lead)) if lead else 1
    packed = np.zeros(lead + (64,), np.uint8)
    scales = np.zeros(lead + (4,), np.uint8)
    _load().orc_quantize_plain(_p(x), n, _p(packed), _p(scales))
    return packed, scales


def dequantize_plain(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    packed, scales = _c(packed, np.uint8), _c(scales, np.uint8)
    lead = packed.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (HEAD_DIM,), np.float64)
    _load().orc_dequantize_plain(_p(packed), _p(scales), n, _p(out))
    return out


def quant_and_cache(k_bf16, slot_mapping, kv_packed: np.ndarray, kv_scale: np.ndarray) -> int:
    """Write tokens into the paged planes in place; returns tokens written or -1 on a bad slot."""
    k = _c(k_bf16, np.uint16)
    s = _c(slot_mapping, np.int32)
    assert kv_packed.flags["C_CONTIGUOUS"] and kv_scale.flags["C_CONTIGUOUS"]
    num_pages = kv_packed.shape[0]
    assert kv_packed.shape[1:] == (4, PAGE, 16) and kv_scale.shape[1:] == (4, PAGE)
    return int(_load().orc_quant_and_cache(_p(k), k.shape[0], _p(s), _p(kv_packed), _p(kv_scale), num_pages))


def read_key(kv_packed, kv_scale, page: int, row: int) -> np.ndarray:
    out = np.zeros(HEAD_DIM, np.float64)
    _load().orc_read_key(_p(kv_packed), _p(kv_scale), int(page), int(row), _p(out))
    return out


# ---- scoring and selection -----------------------------------------------------------

def decode_logits(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, ctx_lens, threads: int = 1):
    q_packed, q_scale = _c(q_packed, np.uint8), _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    bt, ctx = _c(block_tables, np.int32), _c(ctx_lens, np.int32)
    B, H = w.shape
    width = max(int(ctx.max()) if ctx.size else 0, 1)
    out = np.full((B, width), np.nan)
    _load().orc_decode_logits(_p(q_packed), _p(q_scale), _p(w), _p(kv_packed), _p(kv_scale), _p(bt), bt.shape[1],
                              _p(ctx), B, H, _p(out), width, threads)
    return out


def row_logits(q_packed, q_scale, w, r: int, kv_packed, kv_scale, table, t0: int, t1: int):
    q_packed, q_scale = _c(q_packed, np.uint8), _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    table = _c(table, np.int32)
    H = w.shape[1]
    out = np.zeros(max(t1 - t0, 0), np.float64)
    if t1 > t0:
        _load().orc_row_logits(_p(q_packed), _p(q_scale), _p(w), int(r), H, _p(kv_packed), _p(kv_scale), _p(table),
                               int(t0), int(t1), _p(out))
    return out


def prefill_logits(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, cu_seqlens, row_ends, threads: int = 1):
    q_packed, q_scale = _c(q_packed, np.uint8), _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    bt, cu, re = _c(block_tables, np.int32), _c(cu_seqlens, np.int32), _c(row_ends, np.int32)
    R, H = w.shape
    width = max(int(re.max()) if re.size else 0, 1)
    out = np.full((R, width), np.nan)
    _load().orc_prefill_logits(_p(q_packed), _p(q_scale), _p(w), _p(kv_packed), _p(kv_scale), _p(bt), bt.shape[1],
                               _p(cu), _p(re), len(cu) - 1, R, H, _p(out), width, threads)
    return out


def select_topk(logits, n: int, k: int):
    lg = _c(logits, np.float64)
    idx = np.zeros(k, np.int32)
    val = np.zeros(k, np.float64)
    _load().orc_select_topk(_p(lg), int(n), int(k), _p(idx), _p(val))
    return idx, val


def range_topk(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, key_begin, key_end, k: int,
               threads: int = 1):
    """Top-k of each sequence over its keys [key_begin[b], key_end[b]) with absolute indices:
    (topk_idx int32 [B][k], topk_val fp64 [B][k]) in (value desc, index asc) order."""
    q_packed, q_scale = _c(q_packed, np.uint8), _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    bt, kb, ke = _c(block_tables, np.int32), _c(key_begin, np.int32), _c(key_end, np.int32)
    B, H = w.shape
    width = max(int((ke - kb).max()) if kb.size else 0, 1)
    scratch = np.zeros((B, width))
    idx = np.zeros((B, k), np.int32)
    val = np.zeros((B, k), np.float64)
    _load().orc_range_topk(_p(q_packed), _p(q_scale), _p(w), _p(kv_packed), _p(kv_scale), _p(bt), bt.shape[1],
                           _p(kb), _p(ke), B, H, int(k), _p(scratch), width, _p(idx), _p(val), threads)
    return idx, val


def merge_candidates(vals, idx, k: int):
    """Each row's k best of the union of candidate lists vals/idx [lists][rows][k_in] (index < 0
    = empty): (topk_idx int32 [rows][k], topk_val fp64 [rows][k]) in (value desc, index asc) order."""
    vals, idx = _c(vals, np.float64), _c(idx, np.int32)
    L, R, K = idx.shape
    out_idx = np.zeros((R, k), np.int32)
    out_val = np.zeros((R, k), np.float64)
    _load().orc_merge_candidates(_p(vals), _p(idx), L, R, K, int(k), _p(out_idx), _p(out_val))
    return out_idx, out_val


def decode_topk(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, ctx_lens, k: int, threads: int = 1):
    """Returns (topk_idx int32 [B][k], topk_val fp64 [B][k], logits fp64 [B][max_ctx])."""
    q_packed, q_scale = _c(q_packed, np.uint8), _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    bt, ctx = _c(block_tables, np.int32), _c(ctx_lens, np.int32)
    B, H = w.shape
    width = max(int(ctx.max()) if ctx.size else 0, 1)
    scratch = np.full((B, width), np.nan)
    idx = np.zeros((B, k), np.int32)
    val = np.zeros((B, k), np.float64)
    _load().orc_decode_topk(_p(q_packed), _p(q_scale), _p(w), _p(kv_packed), _p(kv_scale), _p(bt), bt.shape[1],
                            _p(ctx), B, H, int(k), _p(scratch), width, _p(idx), _p(val), threads)
    return idx, val, scratch


def prefill_topk(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, cu_seqlens, row_ends, k: int,
                 threads: int = 1):
    q_packed, q_scale = _c(q_packed, np.uint8), _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    bt, cu, re = _c(block_tables, np.int32), _c(cu_seqlens, np.int32), _c(row_ends, np.int32)
    R, H = w.shape
    width = max(int(re.max()) if re.size else 0, 1)
    scratch = np.full((R, width), np.nan)
    idx = np.zeros((R, k), np.int32)
    val = np.zeros((R, k), np.float64)
    _load().orc_prefill_topk(_p(q_packed), _p(q_scale), _p(w), _p(kv_packed), _p(kv_scale), _p(bt), bt.shape[1],
                             _p(cu), _p(re), len(cu) - 1, R, H, int(k), _p(scratch), width, _p(idx), _p(val),
                             threads)
    return idx, val, scratch
