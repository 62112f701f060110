"""The C-ABI library builds, loads, exports every function include/idx_fp4.h declares, and rejects
bad arguments on the host before touching a device (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import fp4_sparse_attention_mxfp4_gb300 as fx
from fp4_sparse_attention_mxfp4_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idx_fp4.h")

OK, ARG, SHAPE, CAP = 0, 1, 2, 3
FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced by these calls
UNALIGNED = ctypes.c_void_p(0x10004)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_fp4_\w+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("idx_fp4_quant_and_cache", "idx_fp4_build_decode_schedule", "idx_fp4_decode_logits_topk",
              "idx_fp4_prefill_logits_topk"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(fx.library_path() if os.path.exists(fx.library_path()) else fx.build_library())
    for name in declared_functions():
        assert hasattr(L, name), f"{name} missing from {fx.library_path()}"
    assert set(declared_functions()) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


@pytest.fixture(scope="module")
def L():
    return _lib.lib()


def test_error_strings(L):
    for code in range(5):
        assert L.idx_fp4_error_string(code)
    assert b"unknown" in L.idx_fp4_error_string(99)


def test_writer_rejects_bad_arguments(L):
    f = L.idx_fp4_quant_and_cache
    assert f(FAKE, -1, FAKE, FAKE, FAKE, 4, None, 0, 0, None, None, None, None) == ARG
    assert f(None, 8, FAKE, FAKE, FAKE, 4, None, 0, 0, None, None, None, None) == ARG
    assert f(UNALIGNED, 8, FAKE, FAKE, FAKE, 4, None, 0, 0, None, None, None, None) == ARG
    assert f(FAKE, 8, FAKE, FAKE, FAKE, 4, FAKE, 2, 48, FAKE, FAKE, None, None) == SHAPE
    assert f(FAKE, 8, FAKE, FAKE, FAKE, 4, FAKE, 2, 64, None, FAKE, None, None) == ARG
    assert f(None, 0, None, None, None, 0, None, 0, 0, None, None, None, None) == OK  # nothing to do


def test_schedule_sizing_and_rejections(L):
    assert L.idx_fp4_decode_schedule_bytes(0, 1 << 20) == 0
    assert L.idx_fp4_decode_schedule_bytes(100000, 1 << 20) == 0
    assert L.idx_fp4_decode_schedule_bytes(16, -1) == 0
    n16 = L.idx_fp4_decode_schedule_bytes(16, 1 << 20)
    assert n16 > 0 and L.idx_fp4_decode_schedule_bytes(32, 1 << 20) > n16
    assert L.idx_fp4_decode_schedule_bytes(16, 1 << 22) > n16
    assert L.idx_fp4_decode_workspace_bytes(16, 1 << 20, 2048) > L.idx_fp4_decode_workspace_bytes(16, 1 << 20, 64)
    assert L.idx_fp4_decode_workspace_bytes(16, 1 << 20, 0) == 0
    f = L.idx_fp4_build_decode_schedule
    assert f(FAKE, 17, 16, 1 << 20, FAKE, n16, None, None) == ARG      # batch > max_batch
    assert f(FAKE, 4, 16, -1, FAKE, n16, None, None) == ARG             # negative max_ctx
    assert f(FAKE, 4, 16, 1 << 20, None, n16, None, None) == ARG        # no buffer
    assert f(FAKE, 4, 16, 1 << 20, UNALIGNED, n16, None, None) == ARG
    assert f(FAKE, 4, 16, 1 << 20, FAKE, n16 - 1, None, None) == CAP    # buffer too small


def _decode(L, **kw):
    a = dict(q=FAKE, qs=FAKE, w=FAKE, kp=FAKE, ks=FAKE, pages=10, bt=FAKE, stride=4, ctx=FAKE, batch=2, heads=64,
             topk=2048, sched=FAKE, sched_bytes=1 << 20, ws=FAKE, ws_bytes=1 << 30, idx=FAKE, val=None, dbg=None,
             dbg_stride=0, status=None, stream=None)
    a.update(kw)
    return L.idx_fp4_decode_logits_topk(*a.values())


def test_decode_rejects_bad_arguments(L):
    assert _decode(L, heads=48) == SHAPE
    assert _decode(L, heads=8) == SHAPE
    assert _decode(L, topk=0) == SHAPE
    assert _decode(L, topk=4096) == SHAPE
    assert _decode(L, batch=-1) == ARG
    assert _decode(L, batch=0) == OK
    assert _decode(L, q=None) == ARG
    assert _decode(L, idx=None) == ARG
    assert _decode(L, sched=None) == ARG
    assert _decode(L, pages=0) == ARG
    assert _decode(L, stride=0) == ARG
    assert _decode(L, dbg=FAKE, dbg_stride=0) == ARG
    assert _decode(L, kp=UNALIGNED) == ARG


def _prefill(L, **kw):
    a = dict(q=FAKE, qs=FAKE, w=FAKE, kp=FAKE, ks=FAKE, pages=10, bt=FAKE, stride=4, ctx=FAKE, cu=FAKE, re=FAKE,
             G=2, R=100, heads=64, topk=2048, max_ctx=4096, ws=FAKE, ws_bytes=1 << 20, idx=FAKE, val=None, dbg=None,
             dbg_stride=0, status=None, stream=None)
    a.update(kw)
    return L.idx_fp4_prefill_logits_topk(*a.values())


def test_prefill_rejects_bad_arguments(L):
    assert _prefill(L, heads=24) == SHAPE
    assert _prefill(L, topk=2049) == SHAPE
    assert _prefill(L, R=0) == OK
    assert _prefill(L, G=0) == ARG
    assert _prefill(L, cu=None) == ARG
    assert _prefill(L, re=None) == ARG
    assert _prefill(L, ws_bytes=16) == CAP
    need = L.idx_fp4_prefill_workspace_bytes(2, 100, 64, 4096, 2048)
    assert need > 0 and _prefill(L, ws_bytes=need - 1) == CAP
    long_need = L.idx_fp4_prefill_workspace_bytes(2, 100, 64, 100000, 2048)
    assert long_need > need  # rows longer than a unit's share need candidate slots
    assert _prefill(L, max_ctx=100000, ws_bytes=need) == CAP
    assert _prefill(L, R=9000) == ARG  # more rows than one call takes
    assert L.idx_fp4_prefill_workspace_bytes(0, 100, 64, 4096, 2048) == 0
    assert L.idx_fp4_prefill_workspace_bytes(2, 100, 48, 4096, 2048) == 0


def test_range_schedule_and_merge_reject_bad_arguments(L):
    n16 = L.idx_fp4_decode_schedule_bytes(16, 1 << 20)
    f = L.idx_fp4_build_decode_schedule_range
    assert f(None, FAKE, 4, 16, 1 << 20, FAKE, n16, None, None) == ARG      # no key_begin
    assert f(FAKE, FAKE, 17, 16, 1 << 20, FAKE, n16, None, None) == ARG     # batch > max_batch
    assert f(FAKE, FAKE, 4, 16, 1 << 20, FAKE, n16 - 1, None, None) == CAP  # buffer too small
    m = L.idx_fp4_merge_candidates
    assert m(FAKE, FAKE, 0, 4, 64, 64, FAKE, None, None, None) == ARG       # no list
    assert m(FAKE, FAKE, 2, -1, 64, 64, FAKE, None, None, None) == ARG      # negative rows
    assert m(FAKE, FAKE, 2, 4, 64, 0, FAKE, None, None, None) == SHAPE      # topk 0
    assert m(FAKE, FAKE, 2, 4, 64, 4096, FAKE, None, None, None) == SHAPE   # topk past the maximum
    assert m(FAKE, FAKE, 9, 4, 2048, 2048, FAKE, None, None, None) == CAP   # 18432 candidates per row
    assert m(FAKE, FAKE, 2, 4, 64, 64, None, None, None, None) == ARG       # no output
    assert m(None, None, 2, 0, 64, 64, None, None, None, None) == OK        # no rows: nothing launched
