// Work schedules for the persistent scorer grid.
//
// Decode ("Score a DSA sparse indexer in FP4", squashed commit message and section "Decode
// grid floor": a persistent-grid CTA schedule built once per step at a CUDA-graph-stable
// address, so a captured graph replays across changing context lengths; a schedule that
// under-covers rows is an error, never silent). The pages size their grid with a fixed floor
// (512 decode / 4096 prefill CTAs) and measure the cost of CTAs past the work. Here the grid
// is the SM count and the work is cut to it: all sequences' 128-key tiles are laid end to end
// and each CTA takes one contiguous, equal share, split at sequence boundaries into units.
// A sequence spread over several units is merged from per-unit candidates afterwards.
//
// Prefill ("Score a DSA sparse indexer in FP4": the prefill scorer finds a row's page table
// through its group and takes per-row key bounds): rows of one request are grouped by
// `rows_per_unit`; a group scores keys [0, max row end) once and masks per row. Groups are
// listed per request from the last (longest) to the first so that a round-robin over CTAs
// starts the longest work first.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace idxfp4 {
namespace {

constexpr int kSchedThreads = 1024;
constexpr int kMaxBatchSched = 4096;

// Exclusive scan of v over the block (kSchedThreads threads, one value each); returns the
// exclusive prefix and writes the total to *total (shared).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    int s = lane < (kSchedThreads / 32) ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, si, off);
      if (lane >= off) si += t;
    }
    warp_sums[lane] = si - s;  // exclusive warp offsets
    if (lane == 31) *total = si;
  }
  __syncthreads();
  const int r = warp_sums[w] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSchedThreads) build_decode_schedule_kernel(const int32_t* __restrict__ ctx_lens,
                                                                              int batch, int max_batch,
                                                                              int64_t max_ctx, int ctas,
                                                                              int min_tiles, void* sched,
                                                                              int32_t* status) {
  __shared__ int s_start[kMaxBatchSched + 1];  // exclusive prefix of tiles per sequence
  __shared__ int s_ne[kMaxBatchSched + 1];     // exclusive prefix of non-empty sequences
  __shared__ int warp_sums[32];
  __shared__ int s_total, s_total_ne, s_scan;
  DecodeSchedView v = decode_sched_view(sched, max_batch);
  const int tid = threadIdx.x;
  constexpr int kPer = kMaxBatchSched / kSchedThreads;  // sequences per thread in the scans

  // 1. tiles per sequence and their prefix sums
  int tiles[kPer], nonempty[kPer];
  int my_tiles = 0, my_ne = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    int c = 0;
    if (b < batch) {
      const int64_t raw = ctx_lens[b];
      if (raw < 0 || raw > max_ctx) {
        set_status(status, IDX_FP4_DEV_BAD_CTX);
      } else {
        c = static_cast<int>(raw);
      }
      v.seq_ctx[b] = c;
    }
    tiles[j] = (c + kTileKeys - 1) / kTileKeys;
    nonempty[j] = tiles[j] > 0 ? 1 : 0;
    my_tiles += tiles[j];
    my_ne += nonempty[j];
  }
  int off = block_exclusive_scan(my_tiles, warp_sums, &s_total);
  int off_ne = block_exclusive_scan(my_ne, warp_sums, &s_total_ne);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    s_start[b] = off;
    s_ne[b] = off_ne;
    off += tiles[j];
    off_ne += nonempty[j];
  }
  if (tid == 0) {
    s_start[kMaxBatchSched] = s_total;
    s_ne[kMaxBatchSched] = s_total_ne;
  }
  __syncthreads();
  const int total = s_total;
  int per = (total + ctas - 1) / ctas;
  if (per < min_tiles) per = min_tiles;
  if (per < 1) per = 1;

  // 2. units per sequence (closed form) and per CTA
  for (int b = tid; b < batch; b += kSchedThreads) {
    const int t = s_start[b + 1] - s_start[b];
    v.seq_units[b] = t > 0 ? ((s_start[b] + t - 1) / per - s_start[b] / per + 1) : 0;
    v.seq_first[b] = -1;
  }
  // seq containing tile x: the last b with start[b] <= x (never an empty sequence)
  auto seq_of = [&](int x) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  int my_count = 0, b0 = 0, b1 = -1, lo_t = 0, hi_t = 0;
  if (tid < ctas) {
    lo_t = tid * per;
    hi_t = min(lo_t + per, total);
    if (lo_t < hi_t) {
      b0 = seq_of(lo_t);
      b1 = seq_of(hi_t - 1);
      my_count = s_ne[b1 + 1] - s_ne[b0];
    }
  }
  __syncthreads();
  const int first = block_exclusive_scan(tid < ctas ? my_count : 0, warp_sums, &s_scan);
  if (tid < ctas) {
    v.cta_first[tid] = first;
    v.cta_count[tid] = my_count;
  }
  __syncthreads();
  // 3. emit units
  if (tid < ctas && my_count > 0) {
    int idx = first;
    for (int b = b0; b <= b1; ++b) {
      const int sb = s_start[b], tb = s_start[b + 1] - sb;
      if (tb == 0) continue;
      const int ulo = max(lo_t, sb), uhi = min(hi_t, sb + tb);
      Unit u;
      u.row = b;
      u.table = b;
      u.kb = (ulo - sb) * kTileKeys;
      u.ke = min((uhi - sb) * kTileKeys, v.seq_ctx[b]);
      u.nq = 1;
      u.slot = v.seq_units[b] == 1 ? -1 : idx;
      u.pad0 = u.pad1 = 0;
      v.units[idx] = u;
      if (ulo == sb) v.seq_first[b] = idx;
      ++idx;
    }
  }
  if (tid == 0) {
    DecodeSchedHeader h;
    h.magic = kDecodeMagic;
    h.ctas = ctas;
    h.batch = batch;
    h.max_batch = max_batch;
    h.num_units = s_scan;
    h.total_tiles = total;
    h.tiles_per_cta = per;
    h.reserved = 0;
    *v.hdr = h;
  }
}

__global__ void __launch_bounds__(kSchedThreads) build_prefill_schedule_kernel(
    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ row_ends,
    const int32_t* __restrict__ ctx_lens, int num_requests, int num_rows, int rows_per_unit, int table_width,
    void* workspace, int32_t* status) {
  __shared__ int warp_sums[32];
  __shared__ int s_total, s_bad;
  __shared__ int s_off[kMaxBatchSched + 1];
  const int tid = threadIdx.x;
  PrefillSchedHeader* hdr = static_cast<PrefillSchedHeader*>(workspace);
  Unit* units = reinterpret_cast<Unit*>(hdr + 1);
  const int Q = rows_per_unit;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // validate cu_seqlens
  for (int g = tid; g < num_requests; g += kSchedThreads) {
    const int a = cu_seqlens[g], b = cu_seqlens[g + 1];
    if (a > b || (g == 0 && a != 0) || (g == num_requests - 1 && b != num_rows)) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    // Rows cannot be mapped to requests: emit empty units over all rows so every row's
    // output is written as "no key", and flag the call.
    if (tid == 0) set_status(status, IDX_FP4_DEV_BAD_ROWS);
    const int n = (num_rows + Q - 1) / Q;
    for (int j = tid; j < n; j += kSchedThreads) {
      Unit u;
      u.row = j * Q;
      u.table = 0;
      u.kb = 0;
      u.ke = 0;
      u.nq = min(Q, num_rows - j * Q);
      u.slot = -1;
      u.pad0 = u.pad1 = 0;
      units[j] = u;
    }
    if (tid == 0) {
      PrefillSchedHeader h{};
      h.magic = kPrefillMagic;
      h.num_units = n;
      h.rows_per_unit = Q;
      *hdr = h;
    }
    return;
  }
  // groups per request and their offsets (requests handled kPer per thread)
  constexpr int kPer = kMaxBatchSched / kSchedThreads;
  int cnt[kPer], my = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int g = tid * kPer + j;
    cnt[j] = g < num_requests ? (cu_seqlens[g + 1] - cu_seqlens[g] + Q - 1) / Q : 0;
    my += cnt[j];
  }
  int off = block_exclusive_scan(my, warp_sums, &s_total);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    s_off[tid * kPer + j] = off;
    off += cnt[j];
  }
  __syncthreads();
  const int total = s_total;
  for (int idx = tid; idx < total; idx += kSchedThreads) {
    // request of unit idx: last g with s_off[g] <= idx and a non-zero count
    int lo = 0, hi = num_requests - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int ng = (cu_seqlens[g + 1] - cu_seqlens[g] + Q - 1) / Q;
    const int j = ng - 1 - (idx - s_off[g]);  // last group first
    const int r0 = cu_seqlens[g] + j * Q;
    const int nq = min(Q, cu_seqlens[g + 1] - r0);
    const int cap = min(ctx_lens[g], table_width * kPage);
    if (ctx_lens[g] < 0) set_status(status, IDX_FP4_DEV_BAD_CTX);
    if (ctx_lens[g] > table_width * kPage) set_status(status, IDX_FP4_DEV_BAD_CTX);
    int ke = 0;
    for (int i = 0; i < nq; ++i) {
      int e = row_ends[r0 + i];
      if (e < 0 || e > cap) {
        set_status(status, IDX_FP4_DEV_BAD_ROWS);
        e = e < 0 ? 0 : cap;
      }
      ke = max(ke, e);
    }
    Unit u;
    u.row = r0;
    u.table = g;
    u.kb = 0;
    u.ke = max(ke, 0);
    u.nq = nq;
    u.slot = -1;
    u.pad0 = u.pad1 = 0;
    units[idx] = u;
  }
  if (tid == 0) {
    PrefillSchedHeader h{};
    h.magic = kPrefillMagic;
    h.num_units = total;
    h.rows_per_unit = Q;
    *hdr = h;
  }
}

}  // namespace

cudaError_t launch_build_decode_schedule(const int32_t* ctx_lens, int batch, int max_batch, int64_t max_ctx, int ctas,
                                         int min_tiles, void* sched, int32_t* status, cudaStream_t stream) {
  build_decode_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(ctx_lens, batch, max_batch, max_ctx, ctas, min_tiles,
                                                                 sched, status);
  return cudaGetLastError();
}

cudaError_t launch_build_prefill_schedule(const int32_t* cu_seqlens, const int32_t* row_ends, const int32_t* ctx_lens,
                                          int num_requests, int num_rows, int rows_per_unit, int table_width,
                                          void* workspace, int32_t* status, cudaStream_t stream) {
  build_prefill_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(cu_seqlens, row_ends, ctx_lens, num_requests,
                                                                  num_rows, rows_per_unit, table_width, workspace,
                                                                  status);
  return cudaGetLastError();
}

int max_batch_supported() { return kMaxBatchSched; }

}  // namespace idxfp4
