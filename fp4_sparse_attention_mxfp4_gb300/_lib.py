"""ctypes binding of libidxfp4.so: argument marshalling only.

Every function here checks tensor dtypes, shapes and devices, passes raw pointers and
sizes to the C ABI (include/idx_fp4.h) and raises on a non-zero return code. All the
work runs in the library's CUDA kernels; there is no Python or CPU fallback, and a
missing or unloadable library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

IDX_FP4_OK = 0
IDX_FP4_ERR_ARG = 1
IDX_FP4_ERR_SHAPE = 2
IDX_FP4_ERR_CAPACITY = 3
IDX_FP4_ERR_CUDA = 4
IDX_FP4_MAX_TOPK = 2048

DEV_BAD_SLOT = 0x01
DEV_BAD_PAGE = 0x02
DEV_BAD_CTX = 0x04
DEV_BAD_ROWS = 0x08
DEV_BAD_SCHEDULE = 0x10
DEV_TIMEOUT = 0x20
DEV_CAPACITY = 0x40
DEV_SYNC = 0x80

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_SZ = ctypes.c_size_t

SIGNATURES = {
    "idx_fp4_quant_and_cache": (_I32, [_P, _I64, _P, _P, _P, _I64, _P, _I64, _I32, _P, _P, _P, _P]),
    "idx_fp4_decode_schedule_bytes": (_SZ, [_I32, _I64]),
    "idx_fp4_build_decode_schedule": (_I32, [_P, _I32, _I32, _I64, _P, _SZ, _P, _P]),
    "idx_fp4_decode_workspace_bytes": (_SZ, [_I32, _I64, _I32]),
    "idx_fp4_decode_logits_topk": (_I32, [_P, _P, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _P, _SZ, _P,
                                          _SZ, _P, _P, _P, _I64, _P, _P]),
    "idx_fp4_build_decode_schedule_mtp": (_I32, [_P, _I32, _I32, _I32, _I64, _P, _SZ, _P, _P]),
    "idx_fp4_decode_mtp_workspace_bytes": (_SZ, [_I32, _I64, _I32, _I32]),
    "idx_fp4_decode_mtp_logits_topk": (_I32, [_P, _P, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32, _P,
                                              _SZ, _P, _SZ, _P, _P, _P, _I64, _P, _P]),
    "idx_fp4_build_decode_schedule_range": (_I32, [_P, _P, _I32, _I32, _I64, _P, _SZ, _P, _P]),
    "idx_fp4_merge_candidates": (_I32, [_P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P]),
    "idx_fp4_mxf4_probe_flops": (_I64, [_I32]),
    "idx_fp4_mxf4_probe": (_I32, [_I32, _P, _P]),
    "idx_fp4_prefill_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I64, _I32]),
    "idx_fp4_decode_static_bytes": (_SZ, [_I32, _I64, _I32]),
    "idx_fp4_decode_logits_topk_static": (_I32, [_P, _P, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I64, _P,
                                                 _SZ, _P, _P, _P, _I64, _P, _P]),
    "idx_fp4_prefill_logits_topk": (_I32, [_P, _P, _P, _P, _P, _I64, _P, _I32, _P, _P, _P, _I32, _I32, _I32, _I32,
                                           _I64, _P, _SZ, _P, _P, _P, _I64, _P, _P]),
    "idx_fp4_error_string": (ctypes.c_char_p, [_I32]),
}


class IdxFp4Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = lib().idx_fp4_error_string(code).decode() if code in (1, 2, 3, 4) else f"code {code}"
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib():
    """Load (building first if the in-tree library is missing or stale) libidxfp4.so."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library missing: {path}")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t):
    # a plain int: the argtypes convert it to void* (no ctypes object per argument)
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:  # the current stream's handle without building a Stream object
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _check(fn: str, code: int):
    if code != IDX_FP4_OK:
        raise IdxFp4Error(fn, code)


def _need(t, name, dtype, ndim=None, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)


def idx_fp4_quant_and_cache(k_bf16, slot_mapping, kv_packed, kv_scale, q_bf16=None, q_packed=None, q_scale=None,
                            status=None, stream=None):
    """Quantise keys [T,128] into the paged cache (slot < 0 skipped); optionally q [R,H,128] -> plain MXFP4."""
    _need(k_bf16, "k_bf16", _BF16, 2)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(kv_packed, "kv_packed", torch.uint8, 4)
    _need(kv_scale, "kv_scale", torch.uint8, 3)
    if k_bf16.shape[1] != 128 or slot_mapping.shape[0] != k_bf16.shape[0]:
        raise ValueError("k_bf16 must be [T,128] with one slot per token")
    if tuple(kv_packed.shape[1:]) != (4, 64, 16) or tuple(kv_scale.shape[1:]) != (4, 64) or \
            kv_scale.shape[0] != kv_packed.shape[0]:
        raise ValueError("cache planes must be [P,4,64,16] and [P,4,64]")
    R = H = 0
    if q_bf16 is not None:
        _need(q_bf16, "q_bf16", _BF16, 3)
        R, H = q_bf16.shape[0], q_bf16.shape[1]
        _need(q_packed, "q_packed", torch.uint8, 3)
        _need(q_scale, "q_scale", torch.uint8, 3)
        if q_bf16.shape[2] != 128 or tuple(q_packed.shape) != (R, H, 64) or tuple(q_scale.shape) != (R, H, 4):
            raise ValueError("q shapes must be [R,H,128] -> [R,H,64] + [R,H,4]")
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_quant_and_cache(_ptr(k_bf16), k_bf16.shape[0], _ptr(slot_mapping), _ptr(kv_packed),
                                         _ptr(kv_scale), kv_packed.shape[0], _ptr(q_bf16), R, H, _ptr(q_packed),
                                         _ptr(q_scale), _ptr(status), _stream(stream))
    _check("idx_fp4_quant_and_cache", code)


def idx_fp4_decode_schedule_bytes(max_batch: int, max_ctx: int) -> int:
    return int(lib().idx_fp4_decode_schedule_bytes(int(max_batch), int(max_ctx)))


def idx_fp4_build_decode_schedule(ctx_lens, max_batch: int, max_ctx: int, sched, status=None, stream=None):
    """Build the decode CTA schedule for ctx_lens (device int32 [B]) into sched (device uint8 buffer)."""
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(sched, "sched", torch.uint8, 1)
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_build_decode_schedule(_ptr(ctx_lens), ctx_lens.shape[0], int(max_batch), int(max_ctx),
                                               _ptr(sched), sched.numel(), _ptr(status), _stream(stream))
    _check("idx_fp4_build_decode_schedule", code)


def idx_fp4_build_decode_schedule_range(key_begin, key_end, max_batch: int, max_ctx: int, sched, status=None,
                                        stream=None):
    """Decode schedule over the key ranges [key_begin[b], key_end[b]) (device int32 [B] each;
    key_begin a multiple of 128). Run the decode call with key_end as its ctx_lens."""
    _need(key_begin, "key_begin", torch.int32, 1)
    _need(key_end, "key_end", torch.int32, 1)
    if key_begin.shape != key_end.shape:
        raise ValueError("key_begin and key_end must have the same shape")
    _need(sched, "sched", torch.uint8, 1)
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_build_decode_schedule_range(_ptr(key_begin), _ptr(key_end), key_end.shape[0], int(max_batch),
                                                     int(max_ctx), _ptr(sched), sched.numel(), _ptr(status),
                                                     _stream(stream))
    _check("idx_fp4_build_decode_schedule_range", code)


def idx_fp4_merge_candidates(cand_val, cand_idx, topk: int, topk_idx, topk_val=None, status=None, stream=None):
    """Exact top-k of the union of candidate lists per row: cand_val f32 / cand_idx int32
    [lists, rows, k_in] (index < 0 = empty) -> topk_idx [rows, topk] (ascending, -1 padded) and
    topk_val (nullable)."""
    _need(cand_val, "cand_val", torch.float32, 3)
    _need(cand_idx, "cand_idx", torch.int32, 3)
    if cand_val.shape != cand_idx.shape:
        raise ValueError("cand_val and cand_idx must have the same shape")
    W, R, K = cand_idx.shape
    _need(topk_idx, "topk_idx", torch.int32, 2)
    if tuple(topk_idx.shape) != (R, int(topk)):
        raise ValueError(f"topk_idx must be [{R}, {topk}]")
    if topk_val is not None:
        _need(topk_val, "topk_val", torch.float32, 2)
        if tuple(topk_val.shape) != (R, int(topk)):
            raise ValueError(f"topk_val must be [{R}, {topk}]")
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_merge_candidates(_ptr(cand_val), _ptr(cand_idx), W, R, K, int(topk), _ptr(topk_idx),
                                          _ptr(topk_val), _ptr(status), _stream(stream))
    _check("idx_fp4_merge_candidates", code)


def idx_fp4_mxf4_probe_flops(iters: int) -> int:
    """FLOPs of one idx_fp4_mxf4_probe launch on the current device."""
    return int(lib().idx_fp4_mxf4_probe_flops(int(iters)))


def idx_fp4_mxf4_probe(iters: int, status=None, stream=None):
    """Launch the MXFP4 MMA rate probe (one CTA per SM, `iters` MMA pairs per issuing warp)."""
    if status is not None:
        _need(status, "status", torch.int32)
    _check("idx_fp4_mxf4_probe", lib().idx_fp4_mxf4_probe(int(iters), _ptr(status), _stream(stream)))


def idx_fp4_decode_workspace_bytes(max_batch: int, max_ctx: int, topk: int) -> int:
    """Workspace bytes of the decode call (zero-fill the buffer once before its first use)."""
    return int(lib().idx_fp4_decode_workspace_bytes(int(max_batch), int(max_ctx), int(topk)))


def idx_fp4_build_decode_schedule_mtp(ctx_lens, next_n: int, max_batch: int, max_ctx: int, sched, status=None,
                                      stream=None):
    """Decode schedule for next_n verify rows per sequence (ctx_lens: device int32 [B])."""
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(sched, "sched", torch.uint8, 1)
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_build_decode_schedule_mtp(_ptr(ctx_lens), ctx_lens.shape[0], int(next_n), int(max_batch),
                                                   int(max_ctx), _ptr(sched), sched.numel(), _ptr(status),
                                                   _stream(stream))
    _check("idx_fp4_build_decode_schedule_mtp", code)


def idx_fp4_decode_mtp_workspace_bytes(max_batch: int, max_ctx: int, topk: int, next_n: int) -> int:
    return int(lib().idx_fp4_decode_mtp_workspace_bytes(int(max_batch), int(max_ctx), int(topk), int(next_n)))


def idx_fp4_decode_mtp_logits_topk(q_packed, q_scale, weights, kv_packed, kv_scale, block_tables, ctx_lens,
                                   next_n: int, topk: int, sched, workspace, topk_idx, topk_val=None,
                                   logits_debug=None, status=None, stream=None):
    """Decode with next_n verify rows per sequence: q rows [B*next_n, H, ...]; row j of sequence b
    sees keys [0, ctx_b - next_n + 1 + j). Writes topk_idx [B*next_n, k] and topk_val."""
    _need(q_packed, "q_packed", torch.uint8, 3)
    R, H = q_packed.shape[0], q_packed.shape[1]
    _need(q_scale, "q_scale", torch.uint8, 3)
    _need(weights, "weights", torch.float32, 2)
    _need(kv_packed, "kv_packed", torch.uint8, 4)
    _need(kv_scale, "kv_scale", torch.uint8, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(sched, "sched", torch.uint8, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    B = ctx_lens.shape[0]
    if R != B * int(next_n) or tuple(q_scale.shape) != (R, H, 4) or tuple(weights.shape) != (R, H) or \
            q_packed.shape[2] != 64:
        raise ValueError("q_packed [B*next_n,H,64], q_scale [B*next_n,H,4], weights [B*next_n,H] expected")
    if block_tables.shape[0] < B or tuple(topk_idx.shape) != (R, topk):
        raise ValueError("block_tables [>=B, W], topk_idx [B*next_n, topk] expected")
    if topk_val is not None:
        _need(topk_val, "topk_val", torch.float32, 2)
        if tuple(topk_val.shape) != (R, topk):
            raise ValueError("topk_val must be [B*next_n, topk]")
    stride = 0
    if logits_debug is not None:
        _need(logits_debug, "logits_debug", torch.float32, 2)
        stride = logits_debug.shape[1]
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_decode_mtp_logits_topk(
        _ptr(q_packed), _ptr(q_scale), _ptr(weights), _ptr(kv_packed), _ptr(kv_scale), kv_packed.shape[0],
        _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), B, int(next_n), H, int(topk), _ptr(sched),
        sched.numel(), _ptr(workspace), workspace.numel(), _ptr(topk_idx), _ptr(topk_val), _ptr(logits_debug),
        stride, _ptr(status), _stream(stream))
    _check("idx_fp4_decode_mtp_logits_topk", code)


def idx_fp4_decode_logits_topk(q_packed, q_scale, weights, kv_packed, kv_scale, block_tables, ctx_lens, topk: int,
                               sched, workspace, topk_idx, topk_val=None, logits_debug=None, status=None,
                               stream=None):
    """Decode scoring + top-k; writes topk_idx [B,k] (ascending token index, -1 padded) and topk_val."""
    _need(q_packed, "q_packed", torch.uint8, 3)
    B, H = q_packed.shape[0], q_packed.shape[1]
    _need(q_scale, "q_scale", torch.uint8, 3)
    _need(weights, "weights", torch.float32, 2)
    _need(kv_packed, "kv_packed", torch.uint8, 4)
    _need(kv_scale, "kv_scale", torch.uint8, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(sched, "sched", torch.uint8, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    if tuple(q_scale.shape) != (B, H, 4) or tuple(weights.shape) != (B, H) or q_packed.shape[2] != 64:
        raise ValueError("q_packed [B,H,64], q_scale [B,H,4], weights [B,H] expected")
    if block_tables.shape[0] < B or ctx_lens.shape[0] != B or tuple(topk_idx.shape) != (B, topk):
        raise ValueError("block_tables [>=B, W], ctx_lens [B], topk_idx [B, topk] expected")
    if topk_val is not None:
        _need(topk_val, "topk_val", torch.float32, 2)
        if tuple(topk_val.shape) != (B, topk):
            raise ValueError("topk_val must be [B, topk]")
    stride = 0
    if logits_debug is not None:
        _need(logits_debug, "logits_debug", torch.float32, 2)
        stride = logits_debug.shape[1]
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_decode_logits_topk(
        _ptr(q_packed), _ptr(q_scale), _ptr(weights), _ptr(kv_packed), _ptr(kv_scale), kv_packed.shape[0],
        _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), B, H, int(topk), _ptr(sched), sched.numel(),
        _ptr(workspace), workspace.numel(), _ptr(topk_idx), _ptr(topk_val), _ptr(logits_debug), stride,
        _ptr(status), _stream(stream))
    _check("idx_fp4_decode_logits_topk", code)


# Bytes of the library's fixed decode scratch array (per GPU).
STATIC_SCRATCH_BYTES = 16 << 20


def idx_fp4_decode_static_bytes(batch: int, max_ctx: int, topk: int) -> int:
    """Scratch bytes idx_fp4_decode_logits_topk_static needs for this batch on the current device."""
    return int(lib().idx_fp4_decode_static_bytes(int(batch), int(max_ctx), int(topk)))


def idx_fp4_decode_logits_topk_static(q_packed, q_scale, weights, kv_packed, kv_scale, block_tables, ctx_lens,
                                      topk: int, max_ctx: int, sched, topk_idx, topk_val=None, logits_debug=None,
                                      status=None, stream=None):
    """Decode scoring + top-k without a workspace argument, for callers that cannot allocate device
    memory: the workspace is a fixed 16 MiB array the library keeps on each GPU. Same outputs as
    idx_fp4_decode_logits_topk. The schedule must be built with max_batch = B and this `max_ctx`.
    Calls that overlap on the GPU share that array and race; the first call on a device should
    come before any stream capture."""
    _need(q_packed, "q_packed", torch.uint8, 3)
    B, H = q_packed.shape[0], q_packed.shape[1]
    _need(q_scale, "q_scale", torch.uint8, 3)
    _need(weights, "weights", torch.float32, 2)
    _need(kv_packed, "kv_packed", torch.uint8, 4)
    _need(kv_scale, "kv_scale", torch.uint8, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(sched, "sched", torch.uint8, 1)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    if tuple(q_scale.shape) != (B, H, 4) or tuple(weights.shape) != (B, H) or q_packed.shape[2] != 64:
        raise ValueError("q_packed [B,H,64], q_scale [B,H,4], weights [B,H] expected")
    if block_tables.shape[0] < B or ctx_lens.shape[0] != B or tuple(topk_idx.shape) != (B, topk):
        raise ValueError("block_tables [>=B, W], ctx_lens [B], topk_idx [B, topk] expected")
    if topk_val is not None:
        _need(topk_val, "topk_val", torch.float32, 2)
        if tuple(topk_val.shape) != (B, topk):
            raise ValueError("topk_val must be [B, topk]")
    stride = 0
    if logits_debug is not None:
        _need(logits_debug, "logits_debug", torch.float32, 2)
        stride = logits_debug.shape[1]
    if status is not None:
        _need(status, "status", torch.int32)
    need = idx_fp4_decode_static_bytes(B, max_ctx, topk) if B > 0 else 0
    if need > STATIC_SCRATCH_BYTES:
        raise ValueError(f"batch {B} x max_ctx {max_ctx} at top-{topk} needs {need} scratch bytes, more than the "
                         f"fixed {STATIC_SCRATCH_BYTES}; split the batch or use idx_fp4_decode_logits_topk")
    code = lib().idx_fp4_decode_logits_topk_static(
        _ptr(q_packed), _ptr(q_scale), _ptr(weights), _ptr(kv_packed), _ptr(kv_scale), kv_packed.shape[0],
        _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), B, H, int(topk), int(max_ctx), _ptr(sched),
        sched.numel(), _ptr(topk_idx), _ptr(topk_val), _ptr(logits_debug), stride, _ptr(status), _stream(stream))
    _check("idx_fp4_decode_logits_topk_static", code)

def idx_fp4_prefill_workspace_bytes(num_requests: int, num_rows: int, num_heads: int, max_ctx: int,
                                    topk: int) -> int:
    return int(lib().idx_fp4_prefill_workspace_bytes(int(num_requests), int(num_rows), int(num_heads), int(max_ctx),
                                                     int(topk)))


def idx_fp4_prefill_logits_topk(q_packed, q_scale, weights, kv_packed, kv_scale, block_tables, ctx_lens, cu_seqlens,
                                row_ends, topk: int, max_ctx: int, workspace, topk_idx, topk_val=None,
                                logits_debug=None, status=None, stream=None):
    """Causal prefill scoring + top-k per row; padding rows (row_end 0) come out all -1. `max_ctx`
    bounds every row end and is the value the workspace was sized with."""
    _need(q_packed, "q_packed", torch.uint8, 3)
    R, H = q_packed.shape[0], q_packed.shape[1]
    _need(q_scale, "q_scale", torch.uint8, 3)
    _need(weights, "weights", torch.float32, 2)
    _need(kv_packed, "kv_packed", torch.uint8, 4)
    _need(kv_scale, "kv_scale", torch.uint8, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(row_ends, "row_ends", torch.int32, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    G = ctx_lens.shape[0]
    if tuple(q_scale.shape) != (R, H, 4) or tuple(weights.shape) != (R, H) or q_packed.shape[2] != 64:
        raise ValueError("q_packed [R,H,64], q_scale [R,H,4], weights [R,H] expected")
    if cu_seqlens.shape[0] != G + 1 or row_ends.shape[0] != R or block_tables.shape[0] < G or \
            tuple(topk_idx.shape) != (R, topk):
        raise ValueError("cu_seqlens [G+1], row_ends [R], block_tables [>=G, W], topk_idx [R, topk] expected")
    if topk_val is not None:
        _need(topk_val, "topk_val", torch.float32, 2)
        if tuple(topk_val.shape) != (R, topk):
            raise ValueError("topk_val must be [R, topk]")
    stride = 0
    if logits_debug is not None:
        _need(logits_debug, "logits_debug", torch.float32, 2)
        stride = logits_debug.shape[1]
    if status is not None:
        _need(status, "status", torch.int32)
    code = lib().idx_fp4_prefill_logits_topk(
        _ptr(q_packed), _ptr(q_scale), _ptr(weights), _ptr(kv_packed), _ptr(kv_scale), kv_packed.shape[0],
        _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), _ptr(cu_seqlens), _ptr(row_ends), G, R, H,
        int(topk), int(max_ctx), _ptr(workspace), workspace.numel(), _ptr(topk_idx), _ptr(topk_val), _ptr(logits_debug), stride,
        _ptr(status), _stream(stream))
    _check("idx_fp4_prefill_logits_topk", code)
