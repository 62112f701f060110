// Block-level exact top-k over ordered 32-bit keys held in shared memory.
//
// The keys of one row (the order-preserving image of its fp32 logits) sit in token order. The
// selection finds the threshold key T (the kk-th largest) with three radix levels (11, 11 and
// 10 bits). The first level's histogram is built while the keys are produced (packed 16-bit
// counters, a few histograms so that warps rarely contend for a word). Passes over the keys
// then list the keys of the threshold's level-1 bin (levels 2 and 3 run on that short list)
// and emit every key above T and the lowest-index keys equal to T, in token order. Ties go to
// the lower token index and the output order is deterministic. Passes read four consecutive
// keys per 16-byte load.
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

// Exclusive block-wide prefix sums of two per-thread counts (thread order). Uses sc[0, 2*NW).
template <int NT>
__device__ __forceinline__ uint2 block_exclusive_scan2(uint32_t a, uint32_t b, uint32_t* sc, int tid, int bar) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t va = __shfl_up_sync(0xFFFFFFFFu, ia, off);
    const uint32_t vb = __shfl_up_sync(0xFFFFFFFFu, ib, off);
    if (lane >= off) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    sc[2 * w] = ia;
    sc[2 * w + 1] = ib;
  }
  named_barrier_sync(bar, NT);
  uint32_t pa = 0, pb = 0;
#pragma unroll
  for (int w2 = 0; w2 < NW; ++w2)
    if (w2 < w) {
      pa += sc[2 * w2];
      pb += sc[2 * w2 + 1];
    }
  named_barrier_sync(bar, NT);
  return make_uint2(pa + ia - a, pb + ib - b);
}

// The run of keys a thread owns in the selection passes: [b0, b1), a multiple of 4 long except
// at the end, runs in thread order. The run length is 4 mod 8 words, so the 16-byte loads of a
// quarter warp fall in distinct banks.
template <int NT>
__device__ __forceinline__ int2 thread_run(int n, int tid) {
  int per = (((n + NT - 1) / NT) + 3) & ~3;
  if ((per & 7) == 0) per += 4;
  const int b0 = min(n, tid * per);
  return make_int2(b0, min(n, b0 + per));
}

// Exact selection of the min(kk, n) largest of n keys (keys[0, n), 16-byte aligned, readable up
// to the next multiple of 4), emitted in token order with ties to the lower index: calls
// emit(keep, out_pos, i, key) for every key i of a run holding kept keys, out_pos dense from 0
// over the kept ones; the callee stores without branching on `keep`. `hw` holds NW_H packed
// level-1 histograms of exactly these keys; once summed it serves as the list of the threshold
// bin's keys (NW_H * 1024 words). Keys must be nonzero (ordered keys of real logits are).
//
// Every pass walks per-thread runs with register counters, and block scans turn the counts into
// list and output offsets: no ballots or atomics sit in the passes' dependence chains, which
// matters with one or two warps per scheduler.
template <int NT, int NW_H, class Emit>
__device__ __forceinline__ void select_topk(const uint32_t* keys, int n, int kk, uint32_t* hw, uint32_t* hist,
                                            uint32_t* sc, int tid, int bar, Emit emit) {
  const int2 run = thread_run<NT>(n, tid);
  uint32_t thr = 0u, need = 0u;  // keep key > thr, and the first `need` keys equal to thr
  uint32_t gtc = 0u, eqc = 0u;   // this run's keys > thr and == thr
  if (kk < n) {
    const uint2 r1 = level1_bin<NT, NW_H>(hw, hist, static_cast<uint32_t>(kk), sc, tid, bar);
    const uint32_t bin = r1.x;
    need = static_cast<uint32_t>(kk) - r1.y;
    const uint32_t in_bin = hist[bin];
    if (in_bin <= static_cast<uint32_t>(NW_H * kHistWords)) {
      // list the bin's keys as (low 21 bits | thread << 21), each run at its scanned offset
      uint32_t* list = hw;
      uint32_t above = 0, inb = 0;
      for (int x = run.x; x < run.y; x += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + x);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t b = key_lane(v, e) >> 21;
          const bool in = x + e < run.y;
          above += (in && b > bin) ? 1u : 0u;
          inb += (in && b == bin) ? 1u : 0u;
        }
      }
      uint32_t off = block_exclusive_scan2<NT>(inb, 0u, sc, tid, bar).x;
      // branch-free: a key outside the bin is written to this lane's spare word of `hist`
      // (unused until the levels below), so lanes never diverge
      uint32_t* spare = hist + (tid & 31);
      if (inb != 0u)
        for (int x = run.x; x < run.y; x += 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(keys + x);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t u = key_lane(v, e);
            const bool hit = x + e < run.y && (u >> 21) == bin;
            *(hit ? list + off : spare) = (u & 0x1FFFFFu) | (static_cast<uint32_t>(tid) << 21);
            off += hit ? 1u : 0u;
          }
        }
      named_barrier_sync(bar, NT);
      const int m = static_cast<int>(in_bin);
      // levels 2 and 3 over the list
      uint32_t low = 0u;
#pragma unroll 1
      for (int level = 0; level < 2; ++level) {
        const int nb = level == 0 ? 2048 : 1024;
        for (int i = tid; i < nb; i += NT) hist[i] = 0u;
        named_barrier_sync(bar, NT);
        for (int x = tid; x < m; x += NT) {
          const uint32_t c = list[x] & 0x1FFFFFu;
          if (level == 0) smem_red_add(&hist[c >> 10], 1u);
          else if ((c >> 10) == (low >> 10)) smem_red_add(&hist[c & 1023u], 1u);
        }
        named_barrier_sync(bar, NT);
        const uint2 r = find_bin<NT>(hist, nb, need, sc, tid, bar);
        need -= r.y;
        low |= level == 0 ? (r.x << 10) : r.x;
      }
      thr = (bin << 21) | low;
      // each run's listed keys above and at the threshold
      for (int i = tid; i < 2 * NT; i += NT) hist[i] = 0u;
      named_barrier_sync(bar, NT);
      for (int x = tid; x < m; x += NT) {
        const uint32_t c = list[x];
        const uint32_t owner = c >> 21, lo = c & 0x1FFFFFu;
        if (lo > low)
          smem_red_add(&hist[owner], 1u);
        else if (lo == low)
          smem_red_add(&hist[NT + owner], 1u);
      }
      named_barrier_sync(bar, NT);
      gtc = above + hist[tid];
      eqc = hist[NT + tid];
    } else {
      auto load4 = [keys](int x) { return *reinterpret_cast<const uint4*>(keys + x); };
      const uint2 th = lower_levels_all<NT>(load4, n, bin << 21, need, hist, sc, tid, bar);
      thr = th.x;
      need = th.y;
      for (int x = run.x; x < run.y; x += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + x);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t u = key_lane(v, e);
          const bool in = x + e < run.y;
          gtc += (in && u > thr) ? 1u : 0u;
          eqc += (in && u == thr) ? 1u : 0u;
        }
      }
    }
  } else {
    gtc = static_cast<uint32_t>(run.y - run.x);
  }
  // output offsets: keys above the threshold, and the equal keys still wanted, of earlier runs
  const uint2 pre = block_exclusive_scan2<NT>(gtc, eqc, sc, tid, bar);
  uint32_t out = pre.x + min(pre.y, need), eqr = pre.y;
  if (gtc + eqc != 0u)
    for (int x = run.x; x < run.y; x += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(keys + x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t u = key_lane(v, e);
        const bool in = x + e < run.y;
        const bool eq = in && u == thr;
        const bool keep = (in && u > thr) || (eq && eqr < need);
        emit(keep, static_cast<int>(out), x + e, u);
        out += keep ? 1u : 0u;
        eqr += eq ? 1u : 0u;
      }
    }
  named_barrier_sync(bar, NT);
}

}  // namespace idxfp4
