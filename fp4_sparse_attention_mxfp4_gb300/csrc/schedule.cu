// Work schedules for the persistent scorer grid.
//
// Decode ("Score a DSA sparse indexer in FP4", squashed commit message and section "Decode
// grid floor": a persistent-grid CTA schedule built once per step at a CUDA-graph-stable
// address, so a captured graph replays across changing context lengths; a schedule that
// under-covers rows is an error, never silent). The pages size their grid with a fixed floor
// (512 decode / 4096 prefill CTAs) and measure the cost of CTAs past the work. Here the grid is
// the SM count and the work is cut to it: all sequences' 128-key tiles are laid end to end,
// cut into ranges of at most unit_key_cap(1) keys whose number is a multiple of the grid, and
// each CTA takes an equal block of consecutive ranges. Ranges split at sequence boundaries
// into units. A sequence spread over several units is merged from per-unit candidates.
//
// Prefill ("Score a DSA sparse indexer in FP4": the prefill scorer finds a row's page table
// through its group and takes per-row key bounds): rows of one request are grouped by
// `rows_per_unit`; a group scores keys [0, max row end) once and masks per row. A group whose
// rows reach past unit_key_cap keys is cut into key chunks whose per-row candidates are merged.
// Groups are listed per request from the last (longest) to the first, so a round-robin over
// CTAs starts the longest work first.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace idxfp4 {
namespace {

constexpr int kSchedThreads = 1024;
constexpr int kPer = kMaxBatch / kSchedThreads;  // sequences (requests) per thread in the scans

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
    const int s = lane < (kSchedThreads / 32) ? warp_sums[lane] : 0;
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
                                                                              int min_tiles, int64_t units_cap,
                                                                              void* sched, int32_t* status) {
  __shared__ int s_start[kMaxBatch + 1];  // exclusive prefix of tiles per sequence
  __shared__ int s_ne[kMaxBatch + 1];     // exclusive prefix of non-empty sequences
  __shared__ int warp_sums[32];
  __shared__ int s_total, s_total_ne, s_scan;
  pdl_wait();
  pdl_trigger();
  DecodeSchedView v = decode_sched_view(sched, max_batch);
  const int tid = threadIdx.x;

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
    s_start[kMaxBatch] = s_total;
    s_ne[kMaxBatch] = s_total_ne;
  }
  __syncthreads();
  const int total = s_total;

  // 2. ranges: `m` per CTA, `per` tiles each (at most a unit's key cap)
  const int cap_tiles = unit_key_cap(1) / kTileKeys;
  const int64_t slab = static_cast<int64_t>(ctas) * cap_tiles;
  const int m = total > 0 ? static_cast<int>((total + slab - 1) / slab) : 1;
  int per = static_cast<int>((static_cast<int64_t>(total) + static_cast<int64_t>(ctas) * m - 1) /
                             (static_cast<int64_t>(ctas) * m));
  if (m == 1 && per < min_tiles) per = min_tiles;
  if (per > cap_tiles) per = cap_tiles;
  if (per < 1) per = 1;
  for (int b = tid; b < batch; b += kSchedThreads) {
    const int t = s_start[b + 1] - s_start[b];
    v.seq_units[b] = t > 0 ? ((s_start[b] + t - 1) / per - s_start[b] / per + 1) : 0;
    v.seq_first[b] = -1;
  }
  // the sequence containing tile x: the last b with start[b] <= x (never an empty one)
  auto seq_of = [&](int x) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // 3. units per CTA
  const int64_t cta_lo = static_cast<int64_t>(tid) * m * per;
  int my_count = 0;
  if (tid < ctas) {
    for (int r = 0; r < m; ++r) {
      const int64_t lo = cta_lo + static_cast<int64_t>(r) * per;
      if (lo >= total) break;
      const int hi = static_cast<int>(lo + per < total ? lo + per : total);
      my_count += s_ne[seq_of(hi - 1) + 1] - s_ne[seq_of(static_cast<int>(lo))];
    }
  }
  __syncthreads();
  const int first = block_exclusive_scan(tid < ctas ? my_count : 0, warp_sums, &s_scan);
  const bool fits = s_scan <= units_cap;
  if (tid < ctas) {
    v.cta_first[tid] = first;
    v.cta_count[tid] = fits ? my_count : 0;
  }
  __syncthreads();
  // 4. emit units in token order
  if (fits && tid < ctas && my_count > 0) {
    int idx = first;
    for (int r = 0; r < m; ++r) {
      const int64_t lo64 = cta_lo + static_cast<int64_t>(r) * per;
      if (lo64 >= total) break;
      const int lo = static_cast<int>(lo64);
      const int hi = lo + per < total ? lo + per : total;
      const int b0 = seq_of(lo), b1 = seq_of(hi - 1);
      for (int b = b0; b <= b1; ++b) {
        const int sb = s_start[b], tb = s_start[b + 1] - sb;
        if (tb == 0) continue;
        const int ulo = max(lo, sb), uhi = min(hi, sb + tb);
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
  }
  if (!fits) {
    // cannot happen when the buffer was sized for (max_batch, max_ctx); report, schedule nothing
    for (int b = tid; b < batch; b += kSchedThreads) v.seq_units[b] = 0;
    if (tid == 0) set_status(status, IDX_FP4_DEV_CAPACITY);
  }
  if (tid == 0) {
    DecodeSchedHeader h;
    h.magic = kDecodeMagic;
    h.ctas = ctas;
    h.batch = batch;
    h.max_batch = max_batch;
    h.num_units = fits ? s_scan : 0;
    h.total_tiles = total;
    h.tiles_per_range = per;
    h.units_cap = static_cast<int32_t>(units_cap);
    *v.hdr = h;
  }
}

constexpr int kMaxPrefillGroups = kMaxPrefillRows + kMaxBatch;

__global__ void __launch_bounds__(kSchedThreads) build_prefill_schedule_kernel(
    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ row_ends,
    const int32_t* __restrict__ ctx_lens, int num_requests, int num_rows, int rows_per_unit, int table_width,
    int64_t units_cap, int64_t slots_cap, void* workspace, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int s_dyn[];
  int* s_off = s_dyn;                   // [kMaxBatch + 1] groups before each request
  int* s_n = s_dyn + kMaxBatch + 1;     // [kMaxPrefillGroups] chunks per group, then unit offsets
  __shared__ int warp_sums[32];
  __shared__ int s_total, s_bad, s_units;
  const int tid = threadIdx.x;
  PrefillSchedHeader* hdr = static_cast<PrefillSchedHeader*>(workspace);
  int4* row_merge = reinterpret_cast<int4*>(hdr + 1);
  Unit* units = reinterpret_cast<Unit*>(static_cast<char*>(workspace) + prefill_units_offset(num_rows));
  const int Q = rows_per_unit;
  const int cap = unit_key_cap(Q);
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int g = tid; g < num_requests; g += kSchedThreads) {
    const int a = cu_seqlens[g], b = cu_seqlens[g + 1];
    if (a > b || (g == 0 && a != 0) || (g == num_requests - 1 && b != num_rows)) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    // Rows cannot be mapped to requests: emit empty units over all rows so every row's output is
    // written as "no key", and flag the call.
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
    for (int r = tid; r < num_rows; r += kSchedThreads) row_merge[r] = make_int4(-1, 1, 0, 0);
    if (tid == 0) {
      PrefillSchedHeader h{};
      h.magic = kPrefillMagic;
      h.num_units = n;
      h.rows_per_unit = Q;
      h.units_cap = static_cast<int32_t>(units_cap);
      h.num_rows = num_rows;
      h.slots_cap = static_cast<int32_t>(slots_cap);
      *hdr = h;
    }
    return;
  }
  // groups per request
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
  const int ngroups = s_total;
  // group idx -> request, first row, rows, and the clamped key end of its longest row
  auto group_info = [&](int idx, int& g, int& r0, int& nq, int& kcap) {
    int lo = 0, hi = num_requests - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    g = lo;
    const int ng = (cu_seqlens[g + 1] - cu_seqlens[g] + Q - 1) / Q;
    const int j = ng - 1 - (idx - s_off[g]);  // last group first
    r0 = cu_seqlens[g] + j * Q;
    nq = min(Q, cu_seqlens[g + 1] - r0);
    kcap = min(max(ctx_lens[g], 0), table_width * kPage);
  };
  // pass 1: key chunks per group
  for (int idx = tid; idx < ngroups; idx += kSchedThreads) {
    int g, r0, nq, kcap;
    group_info(idx, g, r0, nq, kcap);
    if (ctx_lens[g] < 0 || ctx_lens[g] > table_width * kPage) set_status(status, IDX_FP4_DEV_BAD_CTX);
    int ke = 0;
    for (int i = 0; i < nq; ++i) {
      int e = row_ends[r0 + i];
      if (e < 0 || e > kcap) {
        set_status(status, IDX_FP4_DEV_BAD_ROWS);
        e = e < 0 ? 0 : kcap;
      }
      ke = max(ke, e);
    }
    s_n[idx] = ke > cap ? (ke + cap - 1) / cap : 1;
  }
  __syncthreads();
  // pass 2: unit offsets (exclusive scan of the chunk counts, in blocks of the thread count)
  int running = 0;
  for (int base = 0; base < ngroups; base += kSchedThreads) {
    const int idx = base + tid;
    const int n = idx < ngroups ? s_n[idx] : 0;
    const int ex = block_exclusive_scan(n, warp_sums, &s_units);
    if (idx < ngroups) s_n[idx] = running + ex;
    running += s_units;
    __syncthreads();
  }
  const int total_units = running;
  const bool fits = total_units <= units_cap;
  // pass 3: units and the per-row merge table
  for (int idx = tid; idx < ngroups; idx += kSchedThreads) {
    int g, r0, nq, kcap;
    group_info(idx, g, r0, nq, kcap);
    int ends[4] = {0, 0, 0, 0}, ke = 0;
    for (int i = 0; i < nq && i < 4; ++i) {
      ends[i] = min(max(row_ends[r0 + i], 0), kcap);
      ke = max(ke, ends[i]);
    }
    const int nch = ke > cap ? (ke + cap - 1) / cap : 1;
    const int ub = s_n[idx];
    const bool split = nch > 1 && static_cast<int64_t>(ub + nch) * Q <= slots_cap;
    if (nch > 1 && !split) set_status(status, IDX_FP4_DEV_CAPACITY);
    if (fits) {
      for (int c = 0; c < nch; ++c) {
        Unit u;
        u.row = r0;
        u.table = g;
        u.kb = c * cap;
        u.ke = split ? min((c + 1) * cap, ke) : (nch > 1 ? 0 : ke);
        u.nq = nq;
        u.slot = split ? (ub + c) * Q : -1;
        u.pad0 = u.pad1 = 0;
        units[ub + c] = u;
      }
    }
    for (int i = 0; i < nq; ++i) row_merge[r0 + i] = make_int4(split ? ub * Q + i : -1, split ? nch : 1, ends[i], 0);
  }
  if (tid == 0) {
    if (!fits) set_status(status, IDX_FP4_DEV_CAPACITY);
    PrefillSchedHeader h{};
    h.magic = kPrefillMagic;
    h.num_units = fits ? total_units : 0;
    h.rows_per_unit = Q;
    h.units_cap = static_cast<int32_t>(units_cap);
    h.num_rows = num_rows;
    h.slots_cap = static_cast<int32_t>(slots_cap);
    *hdr = h;
  }
}

}  // namespace

cudaError_t launch_build_decode_schedule(const int32_t* ctx_lens, int batch, int max_batch, int64_t max_ctx, int ctas,
                                         int min_tiles, int64_t units_cap, void* sched, int32_t* status,
                                         cudaStream_t stream) {
  return launch_pdl(build_decode_schedule_kernel, dim3(1), dim3(kSchedThreads), 0, stream, 1, ctx_lens, batch,
                    max_batch, max_ctx, ctas, min_tiles, units_cap, sched, status);
}

cudaError_t launch_build_prefill_schedule(const int32_t* cu_seqlens, const int32_t* row_ends, const int32_t* ctx_lens,
                                          int num_requests, int num_rows, int rows_per_unit, int table_width,
                                          int64_t units_cap, int64_t slots_cap, void* workspace, int32_t* status,
                                          cudaStream_t stream) {
  constexpr size_t smem = sizeof(int) * (kMaxBatch + 1 + kMaxPrefillGroups);
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(build_prefill_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  return launch_pdl(build_prefill_schedule_kernel, dim3(1), dim3(kSchedThreads), smem, stream, 1, cu_seqlens,
                    row_ends, ctx_lens, num_requests, num_rows, rows_per_unit, table_width, units_cap, slots_cap,
                    workspace, status);
}

}  // namespace idxfp4
