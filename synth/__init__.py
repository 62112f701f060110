"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no part of the indexer's arithmetic: it draws random numbers,
rounds the drawn fp32 inputs to bf16 (the input dtype), and lays out page tables,
context lengths and prefill chunk schedules. Quantisation, scoring and selection
live only in the CUDA library and, independently, in ``oracle/``.

Generator: splitmix64 over a counter (value i of stream s under seed S is
splitmix64(S * 2^32 + s, i)), Box-Muller for normals. Everything is numpy uint64 /
float64 arithmetic, so a given (seed, stream) yields the same numbers in every
consumer within a process and across runs.

Value recipe (the workloads' stated distributions): q, k ~ N(0, 1) in fp32, with 4
channel indices drawn once per tensor and multiplied by 5 in every row and head
(outlier channels), then rounded to bf16 with round-to-nearest-even; head weights
w ~ N(0, 1) / sqrt(H) in fp32. Pages of a sequence are drawn without replacement
from a pool holding every sequence's pages plus 12.5 % spare pages.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PAGE = 64
HEAD_DIM = 128
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_CHUNK = 1 << 20


def _splitmix64(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        x += _GOLDEN
        z = x
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


class Rng:
    """Counter-based splitmix64 stream; ``fork(i)`` gives an independent sub-stream."""

    def __init__(self, seed: int, stream: int = 0):
        self.seed = int(seed)
        self.stream = int(stream)
        self._ctr = 0

    def fork(self, stream: int) -> "Rng":
        return Rng(self.seed, self.stream * 1000003 + int(stream) + 1)

    def u64(self, n: int) -> np.ndarray:
        base = np.uint64((self.seed * (1 << 32) + self.stream) & ((1 << 64) - 1))
        out = np.empty(n, np.uint64)
        for a in range(0, n, _CHUNK):
            b = min(n, a + _CHUNK)
            with np.errstate(over="ignore"):
                ctr = np.arange(self._ctr + a, self._ctr + b, dtype=np.uint64) * _GOLDEN + base
            out[a:b] = _splitmix64(ctr)
        self._ctr += n
        return out

    def uniform(self, n: int) -> np.ndarray:
        """Uniform doubles in [0, 1) with 53 random bits."""
        return (self.u64(n) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))

    def normal(self, n: int, dtype=np.float64) -> np.ndarray:
        """Box-Muller pairs: element 2i and 2i+1 come from uniforms 2i (radius) and 2i+1 (angle)."""
        m = (n + 1) // 2
        out = np.empty(2 * m, dtype)
        for a in range(0, m, _CHUNK // 2):
            b = min(m, a + _CHUNK // 2)
            u = (self.u64(2 * (b - a)) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))
            r = np.sqrt(-2.0 * np.log(1.0 - u[0::2]))
            t = (2.0 * np.pi) * u[1::2]
            out[2 * a:2 * b:2] = r * np.cos(t)
            out[2 * a + 1:2 * b:2] = r * np.sin(t)
        return out[:n]

    def integers(self, lo: int, hi: int, n: int) -> np.ndarray:
        """Integers in [lo, hi] inclusive."""
        span = np.uint64(hi - lo + 1)
        return (self.u64(n) % span).astype(np.int64) + lo

    def permutation(self, n: int) -> np.ndarray:
        return np.argsort(self.u64(n), kind="stable").astype(np.int64)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = (b + rounding) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def qk_bf16(rng: Rng, lead_shape, outliers: int = 4, factor: float = 5.0) -> np.ndarray:
    """N(0,1) fp32 vectors of HEAD_DIM with `outliers` channels (drawn once per tensor) scaled, as bf16 bits."""
    lead_shape = tuple(int(s) for s in lead_shape)
    n = int(np.prod(lead_shape)) * HEAD_DIM if lead_shape else HEAD_DIM
    x = rng.normal(n, np.float32).reshape(lead_shape + (HEAD_DIM,))
    ch = rng.fork(7).permutation(HEAD_DIM)[:outliers]
    x[..., ch] *= np.float32(factor)
    return bf16_bits(x)


def head_weights(rng: Rng, rows: int, heads: int) -> np.ndarray:
    return (rng.normal(rows * heads) / math.sqrt(heads)).astype(np.float32).reshape(rows, heads)


@dataclasses.dataclass
class PagedLayout:
    num_pages: int
    block_tables: np.ndarray  # int32 [B][max_pages]; unused entries hold `fill`
    seq_pages: list           # per sequence: int64 array of its pages, in logical order

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        """Cache slots (page * 64 + row) of logical tokens [t0, t1) of sequence b."""
        t = np.arange(t0, t1, dtype=np.int64)
        return (self.seq_pages[b][t // PAGE] * PAGE + t % PAGE).astype(np.int32)


def paged_layout(rng: Rng, ctx_lens, spare: float = 0.125, pool_pages: int | None = None,
                 width: int | None = None, fill: int = -1, contiguous: bool = False) -> PagedLayout:
    """Random page tables: each sequence's pages drawn without replacement from one pool. With
    `contiguous`, sequence b takes the pages right after sequence b-1's instead (an identity
    table per sequence over a flat, staged pool)."""
    ctx_lens = [int(c) for c in ctx_lens]
    need = [-(-c // PAGE) for c in ctx_lens]
    total = sum(need)
    num_pages = pool_pages if pool_pages is not None else max(total + int(math.ceil(spare * total)), 1)
    assert num_pages >= total
    perm = np.arange(num_pages) if contiguous else rng.permutation(num_pages)
    width = width if width is not None else max(max(need, default=1), 1)
    bt = np.full((len(ctx_lens), width), fill, np.int32)
    seq_pages, at = [], 0
    for b, n in enumerate(need):
        pages = perm[at:at + n]
        at += n
        bt[b, :n] = pages
        seq_pages.append(pages)
    return PagedLayout(num_pages, bt, seq_pages)


# ---- the workloads -------------------------------------------------------------------

@dataclasses.dataclass
class DecodeCase:
    name: str
    heads: int
    topk: int
    ctx_lens: np.ndarray      # int32 [B]
    layout: PagedLayout
    k_bf16: np.ndarray        # uint16 [sum ctx][128], keys of all sequences in order
    q_bf16: np.ndarray        # uint16 [B][H][128]
    w: np.ndarray             # f32 [B][H]

    @property
    def batch(self):
        return len(self.ctx_lens)

    def all_slots(self) -> np.ndarray:
        return np.concatenate([self.layout.slots(b, 0, int(c)) for b, c in enumerate(self.ctx_lens)]) \
            if self.batch else np.zeros(0, np.int32)


def decode_case(name: str, seed: int, ctx_lens, heads: int, topk: int, pool_pages: int | None = None,
                width: int | None = None) -> DecodeCase:
    rng = Rng(seed)
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    layout = paged_layout(rng.fork(1), ctx, pool_pages=pool_pages, width=width)
    k = qk_bf16(rng.fork(2), (int(ctx.sum()),))
    q = qk_bf16(rng.fork(3), (len(ctx), heads))
    w = head_weights(rng.fork(4), len(ctx), heads)
    return DecodeCase(name, heads, topk, ctx, layout, k, q, w)


def decode_config(n: int) -> DecodeCase:
    """The five decode workloads by number: 1 tiny, 2 batch-1 4K, 3 batch-8 ~128K, 4 (4a) 16x128K, 5 (4b) 8x256K."""
    if n == 1:
        return decode_case("tiny_b2_ctx256-300_h16_k64", 0, [256, 300], 16, 64)
    if n == 2:
        return decode_case("b1_ctx4096_h64_k2048", 1, [4096], 64, 2048, pool_pages=4096)
    if n == 3:
        ctx = Rng(2).fork(9).integers(98304, 131072, 8)
        return decode_case("b8_ctx96k-128k_h64_k2048", 2, ctx, 64, 2048)
    if n == 4:
        return decode_case("b16_ctx131072_h64_k2048", 3, [131072] * 16, 64, 2048)
    if n == 5:
        return decode_case("b8_ctx262144_h64_k2048", 3, [262144] * 8, 64, 2048)
    raise ValueError(n)


def replay_ctx_sets(seed: int, batch: int, max_ctx: int, short_below: int = 2048):
    """Context-length vectors for graph replay: {max}, {U[65536, max]}, {U[1, max]} with its first
    entry drawn below `short_below` (a context shorter than k), then {max} again."""
    r = Rng(seed).fork(11)
    lo = min(65536, max_ctx)
    third = r.fork(1).integers(1, max_ctx, batch).astype(np.int32)
    third[0] = int(r.fork(2).integers(1, max(1, min(short_below, max_ctx) - 1), 1)[0])
    return [np.full(batch, max_ctx, np.int32),
            r.integers(lo, max_ctx, batch).astype(np.int32),
            third,
            np.full(batch, max_ctx, np.int32)]


@dataclasses.dataclass
class PrefillStep:
    rows: int                 # rows of the step including padding rows
    real_rows: int
    cu_seqlens: np.ndarray    # int32 [G+1], requests of this step in order, padding folded into the last
    row_ends: np.ndarray      # int32 [rows]; padding rows carry 0
    requests: np.ndarray      # int64 [G]: request id of each group
    ctx_lens: np.ndarray      # int32 [G]: keys cached for the request once this step's keys are written
    token_ids: np.ndarray     # int64 [real_rows]: global token index (into PrefillCase.k_bf16) of each real row


@dataclasses.dataclass
class PrefillCase:
    name: str
    heads: int
    topk: int
    prompt_lens: np.ndarray   # int32 [num_requests]
    layout: PagedLayout       # one page table row per request
    k_bf16: np.ndarray        # uint16 [sum L][128]
    q_bf16: np.ndarray        # uint16 [sum L][H][128]
    w: np.ndarray             # f32 [sum L][H]
    steps: list

    def token_slots(self) -> np.ndarray:
        return np.concatenate([self.layout.slots(g, 0, int(L)) for g, L in enumerate(self.prompt_lens)])

    def token_request(self):
        starts = np.concatenate([[0], np.cumsum(self.prompt_lens)])
        return starts


def prefill_case(name: str, seed: int, prompt_lens, heads: int, topk: int, budget: int = 512,
                 real_per_step: int = 509, pad_to: int = 8, contiguous: bool = False) -> PrefillCase:
    """Chunked causal prefill: requests processed in order, `real_per_step` real tokens per step (a step
    may span requests), then padding rows up to the next multiple of `pad_to` (at most `budget` rows),
    folded into the step's last request with row_end 0. pad_to=1 disables padding."""
    rng = Rng(seed)
    L = np.asarray(prompt_lens, dtype=np.int32)
    layout = paged_layout(rng.fork(1), L, spare=0.0 if contiguous else 0.125, contiguous=contiguous)
    total = int(L.sum())
    k = qk_bf16(rng.fork(2), (total,))
    q = qk_bf16(rng.fork(3), (total, heads))
    w = head_weights(rng.fork(4), total, heads)
    starts = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    steps = []
    t = 0
    while t < total:
        n = min(real_per_step, total - t)
        toks = np.arange(t, t + n, dtype=np.int64)
        req = np.searchsorted(starts, toks, side="right") - 1
        pos = toks - starts[req]
        groups = []
        for g in np.unique(req):
            sel = req == g
            groups.append((int(g), int(sel.sum()), int(pos[sel].max()) + 1))
        rows = n if pad_to <= 1 else min(budget, -(-n // pad_to) * pad_to)
        pad = rows - n
        cu = [0]
        for _, cnt, _ in groups:
            cu.append(cu[-1] + cnt)
        cu[-1] += pad
        row_ends = np.concatenate([pos + 1, np.zeros(pad, np.int64)]).astype(np.int32)
        steps.append(PrefillStep(rows, n, np.asarray(cu, np.int32), row_ends,
                                 np.asarray([g for g, _, _ in groups], np.int64),
                                 np.asarray([e for _, _, e in groups], np.int32), toks))
        t += n
    return PrefillCase(name, heads, topk, L, layout, k, q, w, steps)


@dataclasses.dataclass
class MtpCase:
    """Decode with next_n query rows per sequence (speculative-decoding verify rows): row j of
    sequence b sees keys [0, ctx_b - next_n + 1 + j)."""
    name: str
    heads: int
    topk: int
    next_n: int
    ctx_lens: np.ndarray      # int32 [B], keys cached per sequence (including the step's next_n)
    layout: PagedLayout
    k_bf16: np.ndarray        # uint16 [sum ctx][128]
    q_bf16: np.ndarray        # uint16 [B * next_n][H][128], rows of sequence b at b * next_n + j
    w: np.ndarray             # f32 [B * next_n][H]

    @property
    def batch(self):
        return len(self.ctx_lens)

    def all_slots(self) -> np.ndarray:
        return np.concatenate([self.layout.slots(b, 0, int(c)) for b, c in enumerate(self.ctx_lens)])

    def row_ends(self) -> np.ndarray:
        j = np.tile(np.arange(self.next_n), self.batch)
        return (np.repeat(self.ctx_lens, self.next_n) - self.next_n + 1 + j).astype(np.int32)

    def cu_seqlens(self) -> np.ndarray:
        return (np.arange(self.batch + 1) * self.next_n).astype(np.int32)


def mtp_case(name: str, seed: int, ctx_lens, heads: int, topk: int, next_n: int) -> MtpCase:
    rng = Rng(seed)
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    assert np.all(ctx >= next_n)
    layout = paged_layout(rng.fork(1), ctx)
    k = qk_bf16(rng.fork(2), (int(ctx.sum()),))
    q = qk_bf16(rng.fork(3), (len(ctx) * next_n, heads))
    w = head_weights(rng.fork(4), len(ctx) * next_n, heads)
    return MtpCase(name, heads, topk, next_n, ctx, layout, k, q, w)


def mtp_config() -> MtpCase:
    """The long-context decode workload with two verify rows per sequence: 16 x 131072 keys,
    next_n 2, 64 heads, topk 2048, seed 6."""
    return mtp_case("mtp2_b16_ctx131072_h64_k2048", 6, [131072] * 16, 64, 2048, 2)


def prefill_flat_config() -> PrefillCase:
    """Prefill over a staged, flat cache: one 16384-token prompt whose pages are consecutive (an
    identity page table), 512-row steps with padding rows, 64 heads, topk 2048, seed 5. Rows past
    8192 keys are scored in key chunks whose candidate lists are merged."""
    return prefill_case("prefill_flat_1req_16384_h64_k2048", 5, [16384], 64, 2048, 512, 509, 8, contiguous=True)


def prefill_config(pad_variant: str = "pad8") -> PrefillCase:
    """Causal prefill workload: 4 prompts ~U[2634, 4295], 512-row steps, 64 heads, topk 2048, seed 4."""
    lens = Rng(4).fork(9).integers(2634, 4295, 4)
    if pad_variant == "pad8":
        return prefill_case("prefill_4req_2634-4295_h64_k2048_pad8", 4, lens, 64, 2048, 512, 509, 8)
    if pad_variant == "odd":
        return prefill_case("prefill_4req_2634-4295_h64_k2048_odd", 4, lens, 64, 2048, 511, 509, 1)
    raise ValueError(pad_variant)
