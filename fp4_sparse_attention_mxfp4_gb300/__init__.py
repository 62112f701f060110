"""MXFP4 DSA lightning indexer for GB300 (sm_103a).

The compute lives in the CUDA library ``libidxfp4.so`` (C ABI in ``include/idx_fp4.h``);
this package is its Python binding plus the build step. Calls take CUDA tensors and run
asynchronously on the current (or given) stream:

    idx_fp4_quant_and_cache        bf16 keys -> paged MXFP4 cache (and q -> plain MXFP4)
    idx_fp4_build_decode_schedule  once per decode step: the persistent-grid work table
    idx_fp4_decode_logits_topk     decode: score every cached key of each sequence, top-k
    idx_fp4_decode_mtp_logits_topk decode with next_n verify rows per sequence (one key pass)
    idx_fp4_prefill_logits_topk    causal prefill: score keys [0, row_end) per row, top-k
    idx_fp4_build_decode_schedule_range  decode over key ranges (a key shard per call)
    idx_fp4_merge_candidates       exact top-k of the union of several shards' candidate lists

``shard.py`` holds the host side of key-sharded decode (ranges per shard, gather, merge).
"""
from ._lib import (  # noqa: F401
    DEV_BAD_CTX,
    DEV_CAPACITY,
    DEV_BAD_PAGE,
    DEV_BAD_ROWS,
    DEV_BAD_SCHEDULE,
    DEV_BAD_SLOT,
    DEV_SYNC,
    DEV_TIMEOUT,
    IDX_FP4_MAX_TOPK,
    IdxFp4Error,
    STATIC_SCRATCH_BYTES,
    idx_fp4_build_decode_schedule,
    idx_fp4_build_decode_schedule_mtp,
    idx_fp4_build_decode_schedule_range,
    idx_fp4_decode_logits_topk,
    idx_fp4_decode_mtp_logits_topk,
    idx_fp4_decode_mtp_workspace_bytes,
    idx_fp4_decode_logits_topk_static,
    idx_fp4_decode_static_bytes,
    idx_fp4_decode_schedule_bytes,
    idx_fp4_decode_workspace_bytes,
    idx_fp4_merge_candidates,
    idx_fp4_mxf4_probe,
    idx_fp4_mxf4_probe_flops,
    idx_fp4_prefill_logits_topk,
    idx_fp4_prefill_workspace_bytes,
    idx_fp4_quant_and_cache,
    lib,
    library_path,
)
from .build import build as build_library  # noqa: F401

PAGE = 64
HEAD_DIM = 128
