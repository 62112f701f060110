// Block-level exact top-k over ordered 32-bit keys held in shared memory.
//
// The keys of one row (the order-preserving image of its fp32 logits) sit in token order. The
// selection finds the threshold key T (the kk-th largest) with three radix levels (11, 11 and
// 10 bits): the first level's histogram is built while the keys are produced (per-warp packed
// 16-bit counters, so warps never contend for a counter), the other two by passes that only
// touch the keys sharing the running prefix. An output pass then emits every key above T and
// the lowest-index keys equal to T, in token order, each warp scanning one contiguous segment.
// Ties go to the lower token index and the output order is deterministic.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace idxfp4 {

// Per-warp level-1 histogram: 2048 bins of a key's top 11 bits, two 16-bit counters per 32-bit
// word (bin b in word b/2, half b%2). A warp counts at most 16384 keys, so halves never carry.
constexpr int kHistWords = 1024;

__device__ __forceinline__ void hist16_add(uint32_t* h, uint32_t key) {
  const uint32_t bin = key >> 21;
  smem_red_add(&h[bin >> 1], 1u << ((bin & 1u) * 16u));
}

// Group-wide search for the bin holding the need-th largest element (1-based) of a histogram of
// `nb` bins (nb a multiple of NT). Returns (bin, count in the bins above it) to every thread.
// Uses sc[0 .. NW+1]; barrier `bar` over NT threads.
template <int NT>
__device__ __forceinline__ uint2 find_bin(const uint32_t* hist, int nb, uint32_t need, uint32_t* sc, int tid,
                                          int bar) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  const int per = nb / NT;
  uint32_t s = 0;
  for (int j = 0; j < per; ++j) s += hist[tid * per + j];
  uint32_t incl = s;  // sum over lanes >= lane of this warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, off);
    if (lane + off < 32) incl += v;
  }
  if (lane == 0) sc[w] = incl;
  named_barrier_sync(bar, NT);
  uint32_t above = incl - s;
  for (int w2 = w + 1; w2 < NW; ++w2) above += sc[w2];
  for (int j = per - 1; j >= 0; --j) {
    const uint32_t c = hist[tid * per + j];
    if (above < need && need <= above + c) {
      sc[NW] = static_cast<uint32_t>(tid * per + j);
      sc[NW + 1] = above;
    }
    above += c;
  }
  named_barrier_sync(bar, NT);
  const uint2 r = make_uint2(sc[NW], sc[NW + 1]);
  named_barrier_sync(bar, NT);
  return r;
}

// Threshold of the kk-th largest of n keys (0 < kk < n), key(i) giving key i. `hw` holds NW_H
// per-warp packed level-1 histograms of exactly these keys; `hist` is 2048 words of scratch.
// Returns (T, need): every key > T is selected, plus the first `need` keys equal to T.
template <int NT, int NW_H, class KeyAt>
__device__ __forceinline__ uint2 radix_threshold(KeyAt key, int n, int kk, const uint32_t* hw, uint32_t* hist, uint32_t* sc,
                                 int tid, int bar) {
  for (int wd = tid; wd < kHistWords; wd += NT) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int w = 0; w < NW_H; ++w) {
      const uint32_t v = hw[w * kHistWords + wd];
      lo += v & 0xFFFFu;
      hi += v >> 16;
    }
    hist[2 * wd] = lo;
    hist[2 * wd + 1] = hi;
  }
  named_barrier_sync(bar, NT);
  uint32_t need = static_cast<uint32_t>(kk);
  uint2 r = find_bin<NT>(hist, 2048, need, sc, tid, bar);
  uint32_t prefix = r.x << 21, mask = 0xFFE00000u;
  need -= r.y;
#pragma unroll 1
  for (int level = 0; level < 2; ++level) {
    const int shift = level == 0 ? 10 : 0;
    const int nb = level == 0 ? 2048 : 1024;
    for (int i = tid; i < nb; i += NT) hist[i] = 0;
    named_barrier_sync(bar, NT);
    for (int i = tid; i < n; i += NT) {
      const uint32_t u = key(i);
      if ((u & mask) == prefix) smem_red_add(&hist[(u >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
    }
    named_barrier_sync(bar, NT);
    r = find_bin<NT>(hist, nb, need, sc, tid, bar);
    prefix |= r.x << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    need -= r.y;
  }
  return make_uint2(prefix, need);
}

// Stable selection output over n keys in token order: keep key > T, and keys == T while fewer
// than `need` of them came before. Calls emit(out_pos, i, key) for every kept key i, out_pos
// dense from 0 in token order. Each warp scans one contiguous segment twice (count, emit).
// Uses sc[0 .. 2*NW-1].
template <int NT, class KeyAt, class Emit>
__device__ __forceinline__ void stable_emit(KeyAt key, int n, uint32_t thr, uint32_t need, uint32_t* sc, int tid, int bar,
                            Emit emit) {
  const int lane = tid & 31, w = tid >> 5;
  const int seg = ((n + NT - 1) / NT) * 32;
  const int b0 = min(n, w * seg), b1 = min(n, b0 + seg);
  uint32_t cg = 0, ce = 0;
  for (int base = b0; base < b1; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < b1 ? key(i) : 0u;
    cg += __popc(__ballot_sync(0xFFFFFFFFu, i < b1 && u > thr));
    ce += __popc(__ballot_sync(0xFFFFFFFFu, i < b1 && u == thr));
  }
  if (lane == 0) {
    sc[2 * w] = cg;
    sc[2 * w + 1] = ce;
  }
  named_barrier_sync(bar, NT);
  uint32_t out = 0, eq_before = 0;
  for (int w2 = 0; w2 < w; ++w2) {
    const uint32_t g = sc[2 * w2], e = sc[2 * w2 + 1];
    out += g + (eq_before >= need ? 0u : min(e, need - eq_before));
    eq_before += e;
  }
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = b0; base < b1; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < b1 ? key(i) : 0u;
    const bool gt = i < b1 && u > thr;
    const bool eq = i < b1 && u == thr;
    const uint32_t beq = __ballot_sync(0xFFFFFFFFu, eq);
    const bool keep = gt || (eq && eq_before + __popc(beq & lt) < need);
    const uint32_t bk = __ballot_sync(0xFFFFFFFFu, keep);
    if (keep) emit(static_cast<int>(out + __popc(bk & lt)), i, u);
    out += __popc(bk);
    eq_before += __popc(beq);
  }
  named_barrier_sync(bar, NT);
}

}  // namespace idxfp4
