// Block-level exact top-k over ordered 32-bit keys held in shared memory.
//
// The keys of one row (the order-preserving image of its fp32 logits) sit in token order. The
// selection finds the threshold key T (the kk-th largest) with three radix levels (11, 11 and
// 10 bits). The first level's histogram is built while the keys are produced (packed 16-bit
// counters, a few histograms so that warps rarely contend for a word). One pass then copies the
// keys of the threshold's level-1 bin into a short list, on which levels 2 and 3 run; a second
// pass emits every key above T and the lowest-index keys equal to T, in token order, each warp
// scanning one contiguous segment. Ties go to the lower token index and the output order is
// deterministic.
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

// Sum of NW_H packed level-1 histograms into hist[0, 2048) and the bin holding the need-th
// largest key: returns (bin, keys in the bins above it). hist keeps the sums.
template <int NT, int NW_H>
__device__ __forceinline__ uint2 level1_bin(const uint32_t* hw, uint32_t* hist, uint32_t need, uint32_t* sc, int tid,
                                            int bar) {
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
  return find_bin<NT>(hist, 2048, need, sc, tid, bar);
}

// Levels 2 and 3 (bits 20..10, then 9..0) over all n keys sharing the level-1 prefix. Returns
// (T, need): the threshold key and how many keys equal to it are still to be taken.
template <int NT, class Load4>
__device__ __forceinline__ uint2 lower_levels_all(Load4 load4, int n, uint32_t prefix, uint32_t need, uint32_t* hist,
                                                  uint32_t* sc, int tid, int bar) {
  uint32_t mask = 0xFFE00000u;
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
    const uint2 r = find_bin<NT>(hist, static_cast<int>(nb), need, sc, tid, bar);
    prefix |= r.x << shift;
    mask |= (nb - 1u) << shift;
    need -= r.y;
  }
  return make_uint2(prefix, need);
}

// Each warp scans one contiguous segment of the n keys: a whole number of 128-key chunks, lane l
// holding keys 4l..4l+3 of a chunk. Segments are in warp order, so warp order is token order.
template <int NT>
__device__ __forceinline__ int2 warp_segment(int n, int w) {
  const int seg = ((n + NT * 4 - 1) / (NT * 4)) * 128;
  const int b0 = min(n, w * seg);
  return make_int2(b0, min(n, b0 + seg));
}

// Per-warp counts of keys > thr (sc[2w]) and == thr (sc[2w+1]) over the warp's segment.
template <int NT, class Load4>
__device__ __forceinline__ void warp_counts(Load4 load4, int n, uint32_t thr, uint32_t* sc, int tid, int bar) {
  const int lane = tid & 31, w = tid >> 5;
  const int2 sg = warp_segment<NT>(n, w);
  uint32_t cg = 0, ce = 0;
#pragma unroll 2
  for (int base = sg.x; base < sg.y; base += 128) {
    const int x = base + 4 * lane;
    if (x < sg.y) {
      const uint4 v = load4(x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t u = key_lane(v, e);
        const bool in = x + e < sg.y;
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
}

// Output pass: keep key > thr, and keys == thr while fewer than `need` of them came before (in
// token order). Calls emit(out_pos, i, key) for every kept key i, out_pos dense from 0 in token
// order. sc[2w], sc[2w+1] hold every warp's counts of keys > thr and == thr in its segment.
template <int NT, class Load4, class Emit>
__device__ __forceinline__ void emit_pass(Load4 load4, int n, uint32_t thr, uint32_t need, const uint32_t* sc, int tid,
                                          int bar, Emit emit) {
  const int lane = tid & 31, w = tid >> 5;
  const int2 sg = warp_segment<NT>(n, w);
  uint32_t out = 0, eq_before = 0;
  for (int w2 = 0; w2 < w; ++w2) {
    const uint32_t g = sc[2 * w2], e = sc[2 * w2 + 1];
    out += g + (eq_before >= need ? 0u : min(e, need - eq_before));
    eq_before += e;
  }
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = sg.x; base < sg.y; base += 128) {
    const int x = base + 4 * lane;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (x < sg.y) v = load4(x);
    uint32_t gtm = 0, eqm = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = key_lane(v, e);
      const bool in = x + e < sg.y;
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

// Threshold search through the level-1 bin alone. One pass over the n keys counts, per warp,
// the keys above the bin and copies the keys inside it into cbuf (the caller has checked that
// they fit) as (low 21 bits | warp << 21). Levels 2 and 3 then run on that short list, and the
// list gives every warp's counts of keys > T and == T, left in sc[2w] and sc[2w+1] for
// emit_pass. Returns (T, need). Uses sc[0, 3*NW + 1].
template <int NT, class Load4>
__device__ __forceinline__ uint2 threshold_in_bin(Load4 load4, int n, uint32_t bin, uint32_t need, uint32_t* cbuf,
                                                  uint32_t* hist, uint32_t* sc, int tid, int bar) {
  constexpr int NW = NT / 32;
  static_assert(NW <= 32, "warp ids fit the list entries");
  const int lane = tid & 31, w = tid >> 5;
  uint32_t* gt1 = sc + 2 * NW;  // per warp: keys above the bin
  uint32_t* cnt = sc + 3 * NW;  // list length
  if (tid == 0) *cnt = 0u;
  named_barrier_sync(bar, NT);
  const int2 sg = warp_segment<NT>(n, w);
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t above = 0;
  for (int base = sg.x; base < sg.y; base += 128) {
    const int x = base + 4 * lane;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (x < sg.y) v = load4(x);
    uint32_t eqm = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = key_lane(v, e);
      const bool in = x + e < sg.y;
      above += (in && (u >> 21) > bin) ? 1u : 0u;
      eqm |= (in && (u >> 21) == bin) ? (1u << e) : 0u;
    }
    uint32_t pre = 0, tot = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, (eqm >> e) & 1u);
      pre += __popc(b & lt);
      tot += __popc(b);
    }
    if (tot != 0u) {
      uint32_t slot = 0;
      if (lane == 0) slot = atomicAdd(cnt, tot);
      slot = __shfl_sync(0xFFFFFFFFu, slot, 0) + pre;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((eqm >> e) & 1u) cbuf[slot++] = (key_lane(v, e) & 0x1FFFFFu) | (static_cast<uint32_t>(w) << 21);
    }
  }
  above = __reduce_add_sync(0xFFFFFFFFu, above);
  if (lane == 0) gt1[w] = above;
  named_barrier_sync(bar, NT);
  const int m = static_cast<int>(*cnt);
  // level 2: bits 20..10 of the listed keys
  for (int i = tid; i < 2048; i += NT) hist[i] = 0u;
  named_barrier_sync(bar, NT);
  for (int x = tid; x < m; x += NT) smem_red_add(&hist[(cbuf[x] & 0x1FFFFFu) >> 10], 1u);
  named_barrier_sync(bar, NT);
  const uint2 r2 = find_bin<NT>(hist, 2048, need, sc, tid, bar);
  need -= r2.y;
  // level 3: bits 9..0 of the listed keys inside that bin
  for (int i = tid; i < 1024; i += NT) hist[i] = 0u;
  named_barrier_sync(bar, NT);
  for (int x = tid; x < m; x += NT) {
    const uint32_t c = cbuf[x] & 0x1FFFFFu;
    if ((c >> 10) == r2.x) smem_red_add(&hist[c & 1023u], 1u);
  }
  named_barrier_sync(bar, NT);
  const uint2 r3 = find_bin<NT>(hist, 1024, need, sc, tid, bar);
  need -= r3.y;
  const uint32_t low = (r2.x << 10) | r3.x;
  // per-warp counts over the list, added to the keys above the bin
  if (tid < NW) {
    sc[2 * tid] = gt1[tid];
    sc[2 * tid + 1] = 0u;
  }
  named_barrier_sync(bar, NT);
  for (int x = tid; x < m; x += NT) {
    const uint32_t c = cbuf[x];
    const uint32_t ww = c >> 21, lo = c & 0x1FFFFFu;
    if (lo > low)
      smem_red_add(&sc[2 * ww], 1u);
    else if (lo == low)
      smem_red_add(&sc[2 * ww + 1], 1u);
  }
  named_barrier_sync(bar, NT);
  return make_uint2((bin << 21) | low, need);
}

// Exact selection of the min(kk, n) largest of n keys, emitted in token order (ties to the lower
// index). `hw` holds NW_H packed level-1 histograms of exactly these keys; once summed it serves
// as the list buffer of threshold_in_bin (NW_H * 1024 words). Keys must be nonzero (ordered keys
// of real logits are), except padding keys 0 that are never wanted.
template <int NT, int NW_H, class Load4, class Emit>
__device__ __forceinline__ void select_topk(Load4 load4, int n, int kk, uint32_t* hw, uint32_t* hist, uint32_t* sc,
                                            int tid, int bar, Emit emit) {
  uint2 th = make_uint2(0u, 0u);  // (T, need): T = 0 keeps every nonzero key
  if (kk < n) {
    const uint2 r1 = level1_bin<NT, NW_H>(hw, hist, static_cast<uint32_t>(kk), sc, tid, bar);
    const uint32_t need = static_cast<uint32_t>(kk) - r1.y;
    if (hist[r1.x] <= static_cast<uint32_t>(NW_H * kHistWords)) {
      th = threshold_in_bin<NT>(load4, n, r1.x, need, hw, hist, sc, tid, bar);
    } else {
      th = lower_levels_all<NT>(load4, n, r1.x << 21, need, hist, sc, tid, bar);
      warp_counts<NT>(load4, n, th.x, sc, tid, bar);
    }
  } else {
    warp_counts<NT>(load4, n, 0u, sc, tid, bar);
  }
  emit_pass<NT>(load4, n, th.x, th.y, sc, tid, bar, emit);
}

}  // namespace idxfp4
