// Prefill work schedule for the persistent scorer grid ("Score a DSA sparse indexer in FP4": the
// prefill scorer finds a row's page table through its group and takes per-row key bounds): rows of
// one request are grouped by `rows_per_unit`; a group scores keys [0, max row end) once and masks
// per row. A group whose rows reach past unit_key_cap keys is cut into key chunks whose per-row
// candidates are merged. Groups are listed per request from the last (longest) to the first, so a
// round-robin over CTAs starts the longest work first.
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

constexpr int kMaxPrefillGroups = kMaxPrefillRows + kMaxBatch;

__device__ __forceinline__ void build_prefill_schedule_body(
    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ row_ends,
    const int32_t* __restrict__ ctx_lens, int num_requests, int num_rows, int rows_per_unit, int table_width,
    int64_t units_cap, int64_t slots_cap, void* workspace, int32_t* status) {
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
    pdl_wait();
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
  // Everything above read only the caller's inputs; the tables below overwrite the workspace that
  // the kernel before this one may still be reading.
  pdl_wait();
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

// The builder reads only its caller's inputs (never what a kernel of this library writes), so it
// starts at once, beside the kernel before it (the writer, when a step runs writer, schedule and
// scorer), and waits for that kernel only before its first write to the workspace: its completion
// still implies its predecessor's, which the scorer launched after it relies on.
__global__ void __launch_bounds__(kSchedThreads) build_prefill_schedule_kernel(
    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ row_ends,
    const int32_t* __restrict__ ctx_lens, int num_requests, int num_rows, int rows_per_unit, int table_width,
    int64_t units_cap, int64_t slots_cap, void* workspace, int32_t* status) {
  pdl_trigger();
  build_prefill_schedule_body(cu_seqlens, row_ends, ctx_lens, num_requests, num_rows, rows_per_unit, table_width,
                              units_cap, slots_cap, workspace, status);
  pdl_wait();
}

}  // namespace

cudaError_t launch_build_prefill_schedule(const int32_t* cu_seqlens, const int32_t* row_ends, const int32_t* ctx_lens,
                                          int num_requests, int num_rows, int rows_per_unit, int table_width,
                                          int64_t units_cap, int64_t slots_cap, void* workspace, int32_t* status,
                                          cudaStream_t stream) {
  constexpr size_t smem = sizeof(int) * (kMaxBatch + 1 + kMaxPrefillGroups);
  cudaError_t e = set_smem_once<build_prefill_schedule_kernel>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(build_prefill_schedule_kernel, dim3(1), dim3(kSchedThreads), smem, stream, 1, false, cu_seqlens,
                    row_ends, ctx_lens, num_requests, num_rows, rows_per_unit, table_width, units_cap, slots_cap,
                    workspace, status);
}

}  // namespace idxfp4
