// Layout constants, device status bits and the work-unit tables shared by the kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <utility>

#include "idx_fp4.h"

namespace idxfp4 {

// Index-cache geometry ("Score a DSA sparse indexer in FP4": index_head_dim 128, page block
// size 64, packed E2M1 plane plus one e8m0 scale per 32 dims).
constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kGroups = 4;                         // scale groups (32 dims each) per key
constexpr int kPageBytes = kGroups * kPage * 16;   // packed plane: [group][row][16 B] = 4096
constexpr int kPageScaleBytes = kGroups * kPage;   // scale plane: [group][swizzled row] = 256
constexpr int kTileKeys = 128;                     // keys per MMA tile (M = 128, two pages)
constexpr int kMaxTopk = IDX_FP4_MAX_TOPK;
constexpr int kMaxCtas = 1024;                     // upper bound on the persistent grid
constexpr int kMaxBatch = 4096;                    // sequences (decode) / requests (prefill) per call
constexpr int kMaxPrefillRows = 8192;              // query rows per prefill call
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: a bound, never reached in normal runs

// Keys one prefill unit scores per query row: the unit's logits live in shared memory (4 B per
// key and row); a unit carries up to two rows.
__host__ __device__ constexpr int unit_key_cap(int rows) { return rows == 1 ? 16384 : 8192; }

// Row permutation of the scale plane inside a page: the 64 rows viewed as 4 x 16 and
// transposed ("Use the index scale plane's own row order when staging FP4 prefill under DCP").
__host__ __device__ constexpr int scale_slot(int row) { return (row % 16) * 4 + row / 16; }

// One unit of prefill scorer work: `nq` query rows sharing one page table, scored against keys
// [kb, ke). kb is a multiple of kTileKeys and ke - kb <= unit_key_cap(rows per unit).
struct Unit {
  int32_t row;    // first query row
  int32_t table;  // row of block_tables
  int32_t kb, ke;
  int32_t nq;
  int32_t slot;   // -1: this unit covers its rows fully and writes the final top-k;
                  // >= 0: candidate slot of its first row (row r uses slot + r), merged afterwards
  int32_t pad0, pad1;
};
static_assert(sizeof(Unit) == 32, "Unit is 32 bytes");

constexpr uint32_t kPrefillMagic = 0x50465332u;  // "PFS2"

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Candidate slots (prefill rows split into key chunks): slot s
// is a 16-byte header (entry count, smallest key, largest key, 0), then up to k
// (ordered key, token index) entries in token order; an odd count is followed by one (0, -1) pad entry so each list
// is a whole number of 16-byte pairs. Key 0 is below every logit's key and never selected.
__host__ __device__ inline size_t cand_slot_entries(int topk) { return round_up(static_cast<size_t>(topk) + 2, 2); }

// Prefill workspace: header | row_merge[num_rows] (first slot, number of lists, clamped row end,
// 0) | (pad to 32) | units[units_cap] | candidate slots[slots_cap]. Row r of a split row group has
// its lists at slots first, first + rows_per_unit, ...; an unsplit row has count 1 and is written
// directly by the scorer.
struct PrefillSchedHeader {
  uint32_t magic;
  int32_t num_units;
  int32_t rows_per_unit;
  int32_t units_cap;
  int32_t num_rows;
  int32_t slots_cap;
  int32_t reserved[2];
};

// Query rows per prefill unit: the MMA N dimension is rows * heads, kept <= 128; each row also
// needs its own logit buffer in shared memory, which caps the count at 2.
__host__ __device__ inline int prefill_rows_per_unit(int heads) { return heads <= 64 ? 2 : 1; }

// Units of a prefill call: one per row group of each request, times the key chunks a row of up
// to max_ctx keys needs.
__host__ __device__ inline int64_t prefill_units_cap(int num_requests, int num_rows, int rows_per_unit,
                                                     int64_t max_ctx) {
  const int64_t groups = (num_rows + rows_per_unit - 1) / rows_per_unit + num_requests;
  const int64_t cap = unit_key_cap(rows_per_unit);
  const int64_t chunks = max_ctx > cap ? (max_ctx + cap - 1) / cap : 1;
  return groups * chunks;
}

__host__ __device__ inline size_t prefill_units_offset(int num_rows) {
  return round_up(sizeof(PrefillSchedHeader) + sizeof(int4) * static_cast<size_t>(num_rows), 32);
}

__host__ __device__ inline size_t prefill_slots_offset(int num_rows, int64_t units_cap) {
  return round_up(prefill_units_offset(num_rows) + sizeof(Unit) * static_cast<size_t>(units_cap), 16);
}

// Candidate slots are only needed by units of split rows; sized for every unit and row.
__host__ __device__ inline size_t prefill_workspace_bytes_for(int num_requests, int num_rows, int rows_per_unit,
                                                               int64_t max_ctx, int topk) {
  const int64_t units = prefill_units_cap(num_requests, num_rows, rows_per_unit, max_ctx);
  const int64_t cap = unit_key_cap(rows_per_unit);
  const int64_t slots = max_ctx > cap ? units * rows_per_unit : 0;
  return prefill_slots_offset(num_rows, units) + sizeof(uint2) * cand_slot_entries(topk) * static_cast<size_t>(slots);
}

// Radix levels of the exact top-k: the first takes the top 12 bits of an ordered key, the next
// two 10 bits each.
constexpr int kL1Bits = 12;
constexpr int kL1Bins = 1 << kL1Bits;
constexpr int kL1Shift = 32 - kL1Bits;

// Order-preserving map fp32 -> uint32 (a larger float maps to a larger integer). Adding
// +0.0f first folds -0 into +0 so that equal values compare equal.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t u) {
  const uint32_t b = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(b);
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// Programmatic dependent launch. Every kernel of this library is launched with programmatic
// stream serialization, so it may begin while the kernel before it in the stream is still
// running, and starts with pdl_wait(): that returns once the preceding grid has completed and
// its memory operations are visible (at once after anything that is not such a kernel). Only
// then does it touch global memory, and only then pdl_trigger() lets the next kernel begin
// launching. Since every kernel waits before it can complete, each completion implies its
// predecessor's, and stream order holds as without the attribute; what is saved is the next
// kernel's launch latency. The schedule builders are the exception: they read only the caller's
// inputs, so they run beside the kernel before them and call pdl_wait() only before their first
// write to global memory other than the status word (their completion still implies their
// predecessor's).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization (plus a cluster shape when cluster_x > 1).
// With `cooperative`, the grid is launched as a cooperative grid: all its CTAs are resident at
// once (the launch fails otherwise), which kernels whose CTAs wait on each other rely on.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              int cluster_x, bool cooperative, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Opt a kernel into `bytes` of dynamic shared memory on the current device, once per device and
// kernel (so that a launch inside stream capture is only a launch). Thread-safe.
template <auto Kernel>
inline cudaError_t set_smem_once(size_t bytes) {
  static std::mutex m;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        static_cast<int>(bytes));
  std::lock_guard<std::mutex> lock(m);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace idxfp4
