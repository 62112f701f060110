// Block-level exact top-k over (ordered key, token index) pairs kept in shared memory.
//
// A candidate buffer holds pairs in ascending token order. Rows stream their logits
// through a threshold filter (a key enters only if it beats the current k-th best);
// when the buffer fills, `block_select` cuts it back to exactly k entries and raises
// the threshold. Selection finds the k-th largest ordered key with three radix passes
// (11/11/10 bits) and then compacts the buffer in place, stably, keeping every key
// above the threshold and the lowest-index keys equal to it. Keeping the buffer in
// token order makes the tie rule exact and the output order deterministic.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace idxfp4 {

// Words of scratch `block_select` needs for a group of NT threads.
template <int NT>
constexpr int select_scratch_words() {
  return (NT / 32) + 2 + 2 * (NT / 32) * 2;
}

// Keep the best `kk` of cb[0, n) (kk < n), stably, by (key desc, position asc). All NT
// threads of the group call it with their group-local `tid`; `hist` holds 2048 words.
// Returns the threshold key (the kk-th largest).
template <int NT>
__device__ uint32_t block_select(uint2* cb, int n, int kk, uint32_t* hist, uint32_t* sc, int tid, int bar_id) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  if (kk <= 0) return 0xFFFFFFFFu;
  uint32_t prefix = 0, mask = 0;
  int need = kk;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < nb; i += NT) hist[i] = 0;
    named_barrier_sync(bar_id, NT);
    for (int i = tid; i < n; i += NT) {
      const uint32_t u = cb[i].x;
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
    }
    named_barrier_sync(bar_id, NT);
    // Thread t owns bins [t*per, (t+1)*per). Find the bin holding the need-th largest key.
    const int per = nb / NT;
    uint32_t s = 0;
    for (int j = 0; j < per; ++j) s += hist[tid * per + j];
    uint32_t incl = s;  // sum over lanes >= lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, off);
      if (lane + off < 32) incl += v;
    }
    if (lane == 0) sc[w] = incl;
    named_barrier_sync(bar_id, NT);
    uint32_t above = incl - s;
    for (int w2 = w + 1; w2 < NW; ++w2) above += sc[w2];
    for (int j = per - 1; j >= 0; --j) {
      const uint32_t c = hist[tid * per + j];
      if (above < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= above + c) {
        sc[NW] = static_cast<uint32_t>(tid * per + j);
        sc[NW + 1] = above;
      }
      above += c;
    }
    named_barrier_sync(bar_id, NT);
    const uint32_t bin = sc[NW];
    need -= static_cast<int>(sc[NW + 1]);
    prefix |= bin << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    named_barrier_sync(bar_id, NT);
  }
  const uint32_t thr = prefix;
  // Stable in-place compaction; round r reads positions [r*NT, r*NT+NT) before any thread
  // writes, and every destination is at or below its source.
  uint32_t* wc_base = sc + NW + 2;
  const uint32_t lt = (1u << lane) - 1u;
  int base = 0, ties = 0, par = 0;
#pragma unroll 1
  for (int start = 0; start < n; start += NT, par ^= 1) {
    const int i = start + tid;
    uint2 e = make_uint2(0u, 0u);
    if (i < n) e = cb[i];
    const bool gt = i < n && e.x > thr;
    const bool eq = i < n && e.x == thr;
    const uint32_t bgt = __ballot_sync(0xFFFFFFFFu, gt), beq = __ballot_sync(0xFFFFFFFFu, eq);
    uint32_t* wc = wc_base + par * NW * 2;
    if (lane == 0) {
      wc[2 * w] = __popc(bgt);
      wc[2 * w + 1] = __popc(beq);
    }
    named_barrier_sync(bar_id, NT);
    int eq_acc = ties, kept_acc = base, my_kept = 0, my_eq = 0;
    for (int w2 = 0; w2 < NW; ++w2) {
      const int g = static_cast<int>(wc[2 * w2]), q = static_cast<int>(wc[2 * w2 + 1]);
      const int keq = max(0, min(q, need - eq_acc));
      if (w2 == w) {
        my_kept = kept_acc;
        my_eq = eq_acc;
      }
      kept_acc += g + keq;
      eq_acc += q;
    }
    const bool keep = gt || (eq && my_eq + __popc(beq & lt) < need);
    const uint32_t bkeep = __ballot_sync(0xFFFFFFFFu, keep);
    if (keep) cb[my_kept + __popc(bkeep & lt)] = e;
    base = kept_acc;
    ties = eq_acc;
  }
  named_barrier_sync(bar_id, NT);
  return thr;
}

// Append up to one pair per thread and row to Q candidate buffers, preserving the order of
// (rank, lane). `wc` holds 2*Q*NW words; `par` alternates per call. One barrier.
template <int Q, int NW>
__device__ __forceinline__ void block_append(uint2* const* cb, int (&count)[Q], const bool (&keep)[Q],
                                             const uint2 (&val)[Q], int rank, int lane, uint32_t* wc, int& par,
                                             int bar_id) {
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t b[Q];
#pragma unroll
  for (int i = 0; i < Q; ++i) {
    b[i] = __ballot_sync(0xFFFFFFFFu, keep[i]);
    if (lane == 0) wc[(par * Q + i) * NW + rank] = __popc(b[i]);
  }
  named_barrier_sync(bar_id, NW * 32);
#pragma unroll
  for (int i = 0; i < Q; ++i) {
    int before = 0, total = 0;
#pragma unroll
    for (int r2 = 0; r2 < NW; ++r2) {
      const int c = static_cast<int>(wc[(par * Q + i) * NW + r2]);
      before += r2 < rank ? c : 0;
      total += c;
    }
    if (keep[i]) cb[i][count[i] + before + __popc(b[i] & lt)] = val[i];
    count[i] += total;
  }
  par ^= 1;
}

}  // namespace idxfp4
