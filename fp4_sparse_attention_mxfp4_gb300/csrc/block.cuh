// Block-wide primitives of the exact top-k: scans, radix histogram searches and an exact
// selection over keys listed in token order. Every block-wide step synchronises on one named
// barrier over the participating threads (the whole CTA in the decode kernel's selection phase).
//
// Keys are the order-preserving 32-bit images of fp32 logits (ordered_key): a larger logit has a
// larger key, equal logits equal keys. Selecting the kk largest keys with ties going to the lower
// token index is then: find the threshold key T (the kk-th largest) and the number `need` of keys
// equal to T that are kept, and keep every key above T plus the first `need` keys equal to T in
// token order. T is found radix-wise, 12 + 10 + 10 bits, with the first level's histogram often
// known beforehand.
#pragma once
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace idxfp4 {

struct Blk {
  int tid, nt;          // thread rank and count (nt a multiple of 32, at most 1024)
  uint32_t bar;         // named barrier over the nt threads
  uint32_t* sc;         // shared scratch, at least 96 words
  __device__ __forceinline__ void sync() const { named_barrier_sync(bar, static_cast<uint32_t>(nt)); }
  __device__ __forceinline__ int lane() const { return tid & 31; }
  __device__ __forceinline__ int warp() const { return tid >> 5; }
  __device__ __forceinline__ int nw() const { return nt >> 5; }
};

// Exclusive prefix (thread order) of two per-thread counts; totals to *ta, *tb.
__device__ __forceinline__ uint2 blk_scan2(const Blk& B, uint32_t a, uint32_t b, uint32_t* ta, uint32_t* tb) {
  const int lane = B.lane(), w = B.warp();
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
    B.sc[2 * w] = ia;
    B.sc[2 * w + 1] = ib;
  }
  B.sync();
  // every warp scans the warp totals across its lanes (lane l holds warp l's)
  uint32_t xa = lane < B.nw() ? B.sc[2 * lane] : 0u, xb = lane < B.nw() ? B.sc[2 * lane + 1] : 0u;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t va = __shfl_up_sync(0xFFFFFFFFu, xa, off);
    const uint32_t vb = __shfl_up_sync(0xFFFFFFFFu, xb, off);
    if (lane >= off) {
      xa += va;
      xb += vb;
    }
  }
  const uint32_t sa = __shfl_sync(0xFFFFFFFFu, xa, 31), sb = __shfl_sync(0xFFFFFFFFu, xb, 31);
  const uint32_t qa = __shfl_sync(0xFFFFFFFFu, xa, w > 0 ? w - 1 : 0);
  const uint32_t qb = __shfl_sync(0xFFFFFFFFu, xb, w > 0 ? w - 1 : 0);
  const uint32_t pa = w > 0 ? qa : 0u, pb = w > 0 ? qb : 0u;
  B.sync();
  if (ta != nullptr) *ta = sa;
  if (tb != nullptr) *tb = sb;
  return make_uint2(pa + ia - a, pb + ib - b);
}

__device__ __forceinline__ void blk_zero(const Blk& B, uint32_t* p, int n) {
  for (int i = B.tid; i < n; i += B.nt) p[i] = 0u;
}

// The contiguous run of [0, n) that thread tid owns in run-based passes (runs in thread order). An
// odd run length puts the lanes of a warp on distinct shared-memory banks in word-wise passes.
__device__ __forceinline__ int2 blk_run(const Blk& B, int n) {
  const int per = ((n + B.nt - 1) / B.nt) | 1;
  const int r0 = min(n, B.tid * per);
  return make_int2(r0, min(n, r0 + per));
}

template <int CB, int FPER>
__device__ __forceinline__ uint2 warp_find_bin2(const uint32_t* fine, const uint32_t* coarse, uint32_t need, int lane);

// The 64 coarse bins of a first-level histogram (coarse c sums fine bins 64c .. 64c + 63), written
// to hist[kL1Bins + c] by warps from the fine bins: one pass over shared memory instead of a second
// atomic per counted key (the keys crowd a few coarse bins, whose atomics would conflict). The
// caller synchronises before and after.
__device__ __forceinline__ void blk_coarse64(const Blk& B, uint32_t* hist) {
  for (int c = B.warp(); c < 64; c += B.nw()) {
    const uint2 v = reinterpret_cast<const uint2*>(hist + c * 64)[B.lane()];
    const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, v.x + v.y);
    if (B.lane() == 0) hist[kL1Bins + c] = sum;
  }
}

// Threshold of an exact top-kk over n candidates whose first-level bin is known: `bin` holds the
// kk-th largest key, and `need` (>= 1) of its keys are among the kk. Finds the low 20 bits of T from
// the keys in `bin`, listed into `list` when they fit list_cap, else counted straight from the
// source in each level. Returns (T, keys equal to T that are kept). key(p) gives candidate p's key.
// *consistent is false when the bin holds fewer than `need` keys (counts that do not belong to
// these candidates); T then keeps nothing from the bin.
template <class KeyAt>
__device__ __forceinline__ uint2 blk_resolve(const Blk& B, KeyAt key, int n, uint32_t bin, uint32_t need,
                                             uint32_t* hist, uint32_t* list, int list_cap, bool* consistent) {
  const int2 run = blk_run(B, n);
  uint32_t cnt = 0;
#pragma unroll 1
  for (int p = run.x; p < run.y; ++p) cnt += (key(p) >> kL1Shift) == bin ? 1u : 0u;
  uint32_t in_bin = 0;
  uint32_t o = blk_scan2(B, cnt, 0u, &in_bin, nullptr).x;
  *consistent = need >= 1u && need <= in_bin;
  if (!*consistent) return make_uint2((bin << kL1Shift) | 0xFFFFFu, 0u);
  const bool listed = in_bin <= static_cast<uint32_t>(list_cap);
  if (listed && cnt != 0u)
#pragma unroll 1
    for (int p = run.x; p < run.y; ++p) {
      const uint32_t k = key(p);
      if ((k >> kL1Shift) == bin) list[o++] = k;
    }
  // two 10-bit levels, each a 1024-bin histogram with 32 coarse bins, searched by one warp
  blk_zero(B, hist, 2 * (1024 + 32));
  B.sync();
  uint32_t low = 0u;
#pragma unroll 1
  for (int level = 0; level < 2; ++level) {
    uint32_t* h = hist + level * (1024 + 32);
    auto count = [&](uint32_t k) {
      if ((k >> kL1Shift) != bin) return;
      const uint32_t l = k & 0xFFFFFu;
      if (level == 1 && (l >> 10) != (low >> 10)) return;
      const uint32_t d = level == 0 ? (l >> 10) : (l & 1023u);
      smem_red_add(&h[d], 1u);
      smem_red_add(&h[1024 + (d >> 5)], 1u);
    };
    if (listed) {
#pragma unroll 1
      for (int i = B.tid; i < static_cast<int>(in_bin); i += B.nt) count(list[i]);
    } else {
#pragma unroll 1
      for (int p = B.tid; p < n; p += B.nt) count(key(p));
    }
    B.sync();
    if (B.warp() == 0) {
      const uint2 r = warp_find_bin2<32, 32>(h, h + 1024, need, B.lane());
      if (B.lane() == 0) {
        B.sc[64] = r.x;
        B.sc[65] = r.y;
      }
    }
    B.sync();
    need -= B.sc[65];
    low |= B.sc[64] << (level == 0 ? 10 : 0);
  }
  return make_uint2((bin << kL1Shift) | low, need);
}

// Bin of the need-th largest element (1 <= need <= total) of hist[0, NB) (NB = 1024 or 4096,
// 16-byte aligned), searched by one warp without block barriers. The bins form 32 groups: a
// coalesced pass sums each group (the lanes reading one group reduce over shuffles) and leaves
// group g's sum in lane g; a suffix scan over the lanes finds the group, and the warp splits that
// group's bins, SUB per lane. Returns (bin, elements in the bins above it) in every lane.
template <int NB>
__device__ __forceinline__ uint2 warp_find_bin(const uint32_t* hist, uint32_t need, int lane) {
  static_assert(NB == 1024 || NB == 4096, "32 groups of 32 or 128 bins");
  constexpr int PER = NB / 32;      // bins per group
  constexpr int G = PER / 4;        // lanes reading one group (16 bytes each)
  constexpr int GCNT = 32 / G;      // groups per pass
  constexpr int SUB = PER / 32;     // bins per lane inside the found group
  const uint4* h4 = reinterpret_cast<const uint4*>(hist);
  uint32_t mine = 0;  // lane g: the sum of group g
#pragma unroll
  for (int it = 0; it < NB / 128; ++it) {
    const uint4 v = h4[it * 32 + lane];
    uint32_t x = v.x + v.y + v.z + v.w;
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    const int gfirst = it * GCNT;
    const uint32_t y = __shfl_sync(0xFFFFFFFFu, x, ((lane - gfirst) & (GCNT - 1)) * G);
    if (lane >= gfirst && lane < gfirst + GCNT) mine = y;
  }
  uint32_t suf = mine;  // elements in groups >= lane
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf, off);
    if (lane + off < 32) suf += t;
  }
  const unsigned m = __ballot_sync(0xFFFFFFFFu, suf - mine < need && need <= suf);
  const int L = m != 0u ? 31 - __clz(m) : 0;
  const uint32_t above_l = __shfl_sync(0xFFFFFFFFu, suf - mine, L);
  uint32_t c[SUB], s2 = 0;
  if constexpr (SUB == 4) {
    const uint4 v = h4[L * 32 + lane];
    c[0] = v.x;
    c[1] = v.y;
    c[2] = v.z;
    c[3] = v.w;
  } else {
    c[0] = hist[L * PER + lane];
  }
#pragma unroll
  for (int k = 0; k < SUB; ++k) s2 += c[k];
  uint32_t suf2 = s2;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf2, off);
    if (lane + off < 32) suf2 += t;
  }
  const uint32_t a2 = above_l + suf2 - s2;
  const unsigned m2 = __ballot_sync(0xFFFFFFFFu, a2 < need && need <= a2 + s2);
  const int L2 = m2 != 0u ? 31 - __clz(m2) : 0;
  uint32_t bin = 0, ab = 0;
  if (lane == L2) {
    uint32_t a = a2;
#pragma unroll
    for (int k = SUB - 1; k >= 0; --k) {
      if (a < need && need <= a + c[k]) {
        bin = static_cast<uint32_t>(L * PER + lane * SUB + k);
        ab = a;
      }
      a += c[k];
    }
  }
  return make_uint2(__shfl_sync(0xFFFFFFFFu, bin, L2), __shfl_sync(0xFFFFFFFFu, ab, L2));
}

// Element e of a 16-byte vector of keys.
__device__ __forceinline__ uint32_t vec_lane(const uint4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// Bin of the need-th largest element (1 <= need <= total) of a two-level histogram, by one warp:
// coarse[c] sums fine[c * FPER, (c + 1) * FPER), CB coarse bins (32 or 64). The warp finds the
// coarse bin from the top, then the fine bin inside it (each lane holding CB / 32 and FPER / 32
// bins). Returns (fine bin, elements above it) in every lane.
template <int CB, int FPER>
__device__ __forceinline__ uint2 warp_find_bin2(const uint32_t* fine, const uint32_t* coarse, uint32_t need, int lane) {
  static_assert((CB == 32 || CB == 64) && (FPER == 32 || FPER == 64), "one or two bins per lane");
  // One level: lane l holds bins PER*l .. PER*l + PER - 1 of h; returns the bin holding the need-th
  // largest element and the elements above it (above0: elements above h's first bin... last bin).
  auto search = [lane, need](const uint32_t* h, auto per_c, uint32_t above0) {
    constexpr int PER = decltype(per_c)::value;
    uint32_t c0, c1 = 0u;
    if constexpr (PER == 2) {
      const uint2 v = reinterpret_cast<const uint2*>(h)[lane];
      c0 = v.x;
      c1 = v.y;
    } else {
      c0 = h[lane];
    }
    const uint32_t s = c0 + c1;
    uint32_t suf = s;  // elements in this lane's bins and above
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf, off);
      if (lane + off < 32) suf += t;
    }
    const uint32_t a = above0 + suf - s;  // elements above this lane's bins
    const unsigned m = __ballot_sync(0xFFFFFFFFu, a < need && need <= a + s);
    const int L = m != 0u ? 31 - __clz(m) : 0;
    // inside lane L: the upper bin first
    const bool hi = PER == 2 && a < need && need <= a + c1;
    const uint32_t bin = static_cast<uint32_t>(lane * PER + (PER == 2 && !hi ? 0 : PER - 1));
    const uint32_t ab = PER == 2 && !hi ? a + c1 : a;
    return make_uint2(__shfl_sync(0xFFFFFFFFu, bin, L), __shfl_sync(0xFFFFFFFFu, ab, L));
  };
  const uint2 c = search(coarse, std::integral_constant<int, CB / 32>{}, 0u);
  const uint2 f = search(fine + c.x * FPER, std::integral_constant<int, FPER / 32>{}, c.y);
  return make_uint2(c.x * FPER + f.x, f.y);
}

// The run of [0, n) that thread tid owns in run-based passes over 16-byte aligned keys: a multiple
// of 4 long (except the last), runs in thread order. A run length of 4 mod 8 words spreads the 16-byte
// loads of a warp's lanes over every bank.
__device__ __forceinline__ int2 blk_run4(const Blk& B, int n) {
  int per = (((n + B.nt - 1) / B.nt) + 3) & ~3;
  if ((per & 7) == 0) per += 4;
  const int r0 = min(n, B.tid * per);
  return make_int2(r0, min(n, r0 + per));
}

}  // namespace idxfp4
