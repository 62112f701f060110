// Block-level exact top-k over ordered 32-bit keys held in shared memory.
//
// The keys of one row (the order-preserving image of its fp32 logits) sit in token order. The
// selection finds the threshold key T (the kk-th largest) with three radix levels (11, 11 and
// 10 bits): the first level's histogram is built while the keys are produced (packed 16-bit
// counters, a few histograms so that warps rarely contend for a word), the other two by passes
// that only count the keys sharing the running prefix. An output pass then emits every key
// above T and the lowest-index keys equal to T, in token order, each warp scanning one
// contiguous segment. Ties go to the lower token index and the output order is deterministic.
//
// Every pass reads four consecutive keys per thread and load (`load4(x)` for x a multiple of
// 4), so each thread keeps several independent shared-memory loads in flight: with one or two
// warps per scheduler, a pass that waited on one key at a time would be bound by load latency.
// Callers guarantee that reading keys [x, x + 4) is in bounds for every x < n.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace idxfp4 {

// Level-1 histogram: 2048 bins of a key's top 11 bits, two 16-bit counters per 32-bit word
// (bin b in word b/2, half b%2). A histogram counts fewer than 65536 keys, so halves never carry.
constexpr int kHistWords = 1024;

__device__ __forceinline__ void hist16_add(uint32_t* h, uint32_t key) {
  const uint32_t bin = key >> 21;
  smem_red_add(&h[bin >> 1], 1u << ((bin & 1u) * 16u));
}

__device__ __forceinline__ uint32_t key_lane(const uint4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
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

// Threshold of the kk-th largest of n keys (0 < kk < n). `hw` holds NW_H packed level-1
// histograms whose sum counts exactly these keys; `hist` is 2048 words of scratch.
// Returns (T, need): every key > T is selected, plus the first `need` keys equal to T.
template <int NT, int NW_H, class Load4>
__device__ __forceinline__ uint2 radix_threshold(Load4 load4, int n, int kk, const uint32_t* hw, uint32_t* hist,
                                                 uint32_t* sc, int tid, int bar) {
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
    const uint32_t nb = level == 0 ? 2048u : 1024u;
    for (int i = tid; i < static_cast<int>(nb); i += NT) hist[i] = 0;
    named_barrier_sync(bar, NT);
#pragma unroll 2
    for (int x = tid * 4; x < n; x += NT * 4) {
      const uint4 v = load4(x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t u = key_lane(v, e);
        if (x + e < n && (u & mask) == prefix) smem_red_add(&hist[(u >> shift) & (nb - 1u)], 1u);
      }
    }
    named_barrier_sync(bar, NT);
    r = find_bin<NT>(hist, static_cast<int>(nb), need, sc, tid, bar);
    prefix |= r.x << shift;
    mask |= (nb - 1u) << shift;
    need -= r.y;
  }
  return make_uint2(prefix, need);
}

// Stable selection output over n keys in token order: keep key > T, and keys == T while fewer
// than `need` of them came before. Calls emit(out_pos, i, key) for every kept key i, out_pos
// dense from 0 in token order. Each warp scans one contiguous segment (a whole number of
// 128-key chunks, lane l holding keys 4l..4l+3 of a chunk) twice: count, then emit.
// Uses sc[0 .. 2*NW-1].
template <int NT, class Load4, class Emit>
__device__ __forceinline__ void stable_emit(Load4 load4, int n, uint32_t thr, uint32_t need, uint32_t* sc, int tid,
                                            int bar, Emit emit) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  const int seg = ((n + NT * 4 - 1) / (NT * 4)) * 128;
  const int b0 = min(n, w * seg), b1 = min(n, b0 + seg);
  uint32_t cg = 0, ce = 0;
#pragma unroll 2
  for (int base = b0; base < b1; base += 128) {
    const int x = base + 4 * lane;
    if (x < b1) {
      const uint4 v = load4(x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t u = key_lane(v, e);
        const bool in = x + e < b1;
        cg += (in && u > thr) ? 1u : 0u;
        ce += (in && u == thr) ? 1u : 0u;
      }
    }
  }
  cg = __reduce_add_sync(0xFFFFFFFFu, cg);
  ce = __reduce_add_sync(0xFFFFFFFFu, ce);
  if (lane == 0) {
    sc[2 * w] = cg;
    sc[2 * w + 1] = ce;
  }
  named_barrier_sync(bar, NT);
  uint32_t out = 0, eq_before = 0;
  for (int w2 = 0; w2 < w && w2 < NW; ++w2) {
    const uint32_t g = sc[2 * w2], e = sc[2 * w2 + 1];
    out += g + (eq_before >= need ? 0u : min(e, need - eq_before));
    eq_before += e;
  }
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = b0; base < b1; base += 128) {
    const int x = base + 4 * lane;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (x < b1) v = load4(x);
    uint32_t gtm = 0, eqm = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = key_lane(v, e);
      const bool in = x + e < b1;
      gtm |= (in && u > thr) ? (1u << e) : 0u;
      eqm |= (in && u == thr) ? (1u << e) : 0u;
    }
    // equal keys in earlier lanes of this chunk
    uint32_t eq_lanes = 0, eq_chunk = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, (eqm >> e) & 1u);
      eq_lanes += __popc(b & lt);
      eq_chunk += __popc(b);
    }
    uint32_t keepm = 0;
    uint32_t rank = eq_before + eq_lanes;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool eq = (eqm >> e) & 1u;
      const bool keep = ((gtm >> e) & 1u) || (eq && rank < need);
      keepm |= keep ? (1u << e) : 0u;
      rank += eq ? 1u : 0u;
    }
    uint32_t k_lanes = 0, k_chunk = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, (keepm >> e) & 1u);
      k_lanes += __popc(b & lt);
      k_chunk += __popc(b);
    }
    uint32_t pos = out + k_lanes;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((keepm >> e) & 1u) {
        emit(static_cast<int>(pos), x + e, key_lane(v, e));
        ++pos;
      }
    }
    out += k_chunk;
    eq_before += eq_chunk;
  }
  named_barrier_sync(bar, NT);
}

}  // namespace idxfp4
