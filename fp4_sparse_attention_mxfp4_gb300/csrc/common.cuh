// Layout constants, device status bits and the work-unit tables shared by the kernels.
#pragma once
#include <cstdint>

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
constexpr int kCandCap = 2 * kMaxTopk + 256;       // per-row candidate buffer (entries)
constexpr int kMaxCtas = 1024;                     // upper bound on the persistent grid
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: a bound, never reached in normal runs

// Row permutation of the scale plane inside a page: the 64 rows viewed as 4 x 16 and
// transposed ("Use the index scale plane's own row order when staging FP4 prefill under DCP").
__host__ __device__ constexpr int scale_slot(int row) { return (row % 16) * 4 + row / 16; }

// One unit of scorer work: `nq` query rows sharing one page table, scored against keys
// [kb, ke). kb is a multiple of kTileKeys.
struct Unit {
  int32_t row;    // first query row (decode: the sequence)
  int32_t table;  // row of block_tables
  int32_t kb, ke;
  int32_t nq;
  int32_t slot;   // -1: this unit covers its rows fully and writes the final top-k;
                  // >= 0: candidate slot in the decode workspace (merged afterwards)
  int32_t pad0, pad1;
};
static_assert(sizeof(Unit) == 32, "Unit is 32 bytes");

constexpr uint32_t kDecodeMagic = 0x44534331u;   // "DSC1"
constexpr uint32_t kPrefillMagic = 0x50465331u;  // "PFS1"

// Decode schedule, at a fixed address the caller owns (CUDA-graph stable):
//   header | cta_first[kMaxCtas] | cta_count[kMaxCtas] | seq_first[max_batch] |
//   seq_units[max_batch] | seq_ctx[max_batch] | (pad to 32) | units[kMaxCtas + max_batch]
struct DecodeSchedHeader {
  uint32_t magic;
  int32_t ctas;         // persistent grid the schedule was built for
  int32_t batch;
  int32_t max_batch;
  int32_t num_units;
  int32_t total_tiles;
  int32_t tiles_per_cta;
  int32_t reserved;
};

struct DecodeSchedView {
  DecodeSchedHeader* hdr;
  int32_t* cta_first;
  int32_t* cta_count;
  int32_t* seq_first;
  int32_t* seq_units;
  int32_t* seq_ctx;
  Unit* units;
};

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t decode_sched_bytes(int max_batch) {
  size_t b = sizeof(DecodeSchedHeader) + 2 * sizeof(int32_t) * kMaxCtas + 3 * sizeof(int32_t) * max_batch;
  b = round_up(b, 32);
  return b + sizeof(Unit) * (kMaxCtas + static_cast<size_t>(max_batch));
}

__host__ __device__ inline DecodeSchedView decode_sched_view(void* base, int max_batch) {
  DecodeSchedView v;
  char* p = static_cast<char*>(base);
  v.hdr = reinterpret_cast<DecodeSchedHeader*>(p);
  p += sizeof(DecodeSchedHeader);
  v.cta_first = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * kMaxCtas;
  v.cta_count = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * kMaxCtas;
  v.seq_first = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * max_batch;
  v.seq_units = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * max_batch;
  v.seq_ctx = reinterpret_cast<int32_t*>(p);
  size_t off = round_up(sizeof(DecodeSchedHeader) + 2 * sizeof(int32_t) * kMaxCtas + 3 * sizeof(int32_t) * max_batch,
                        32);
  v.units = reinterpret_cast<Unit*>(static_cast<char*>(base) + off);
  return v;
}

// Decode workspace: candidates of split sequences, one slot per unit:
//   cand_count[slots] (padded to 16 B) | cand[slots][topk] as (ordered key, token index)
__host__ __device__ inline size_t decode_workspace_bytes_for(int slots, int topk) {
  return round_up(sizeof(int32_t) * slots, 16) + sizeof(uint2) * static_cast<size_t>(slots) * topk;
}

// Prefill workspace: header + unit table.
struct PrefillSchedHeader {
  uint32_t magic;
  int32_t num_units;
  int32_t rows_per_unit;
  int32_t reserved[5];
};

__host__ __device__ inline int prefill_max_units(int num_requests, int num_rows, int rows_per_unit) {
  return (num_rows + rows_per_unit - 1) / rows_per_unit + num_requests;
}

__host__ __device__ inline size_t prefill_workspace_bytes_for(int num_requests, int num_rows, int rows_per_unit) {
  return sizeof(PrefillSchedHeader) + sizeof(Unit) * static_cast<size_t>(prefill_max_units(num_requests, num_rows,
                                                                                             rows_per_unit));
}

// Query rows per prefill unit: the MMA N dimension is rows * heads, kept <= 128; each row
// also needs its own candidate buffer in shared memory, which caps the count at 2.
__host__ __device__ inline int prefill_rows_per_unit(int heads) { return heads <= 64 ? 2 : 1; }

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

}  // namespace idxfp4
