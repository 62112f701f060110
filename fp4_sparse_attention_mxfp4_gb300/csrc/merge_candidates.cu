// Merge of per-shard candidate lists ("Score a DSA sparse indexer in FP4", section "Decode context
// parallelism": each rank scores its own shard of a sequence's keys, keeps its local top-k, and the
// ranks' candidates are gathered and merged into the row's top-k). One CTA per row takes the row's
// candidates from every list, ranks them by (value descending, token ascending), keeps the best
// min(topk, valid candidates) and writes them in ascending token order, padded with -1 / -inf.
//
// A row holds at most IDX_FP4_MERGE_MAX_CANDIDATES candidates (lists x per-list length), so both
// orderings are bitonic sorts in shared memory: 64-bit words (ordered value << 32 | ~token)
// descending, then the kept tokens (token << 32 | ordered value) ascending. Entries whose token is
// negative are empty.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace idxfp4 {
namespace {

constexpr int kMergeThreads = 1024;

// Bitonic sort of s[0, n) (n a power of two), ascending or descending, over the whole block.
__device__ void block_bitonic_sort(uint64_t* s, int n, bool descending) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (n >> 1); t += blockDim.x) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0) != descending;  // this pair's direction
        const uint64_t a = s[lo], b = s[hi];
        if ((a > b) == up) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kMergeThreads) merge_candidates_kernel(
    const float* __restrict__ cand_val, const int32_t* __restrict__ cand_idx, int lists, int rows, int k_in, int topk,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_val) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint64_t s_words[];
  __shared__ int s_valid;
  const int row = blockIdx.x;
  const int n = lists * k_in;
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  uint64_t* s_rank = s_words;       // [n2] candidates by (value desc, token asc)
  uint64_t* s_tok = s_words + n2;   // [k2] the kept ones by token
  if (threadIdx.x == 0) s_valid = 0;
  __syncthreads();
  int mine = 0;
  for (int x = threadIdx.x; x < n2; x += blockDim.x) {
    uint64_t w = 0;  // empty: below every candidate
    if (x < n) {
      const int l = x / k_in, i = x - l * k_in;
      const int64_t at = (static_cast<int64_t>(l) * rows + row) * k_in + i;
      const int32_t t = cand_idx[at];
      if (t >= 0) {
        w = (static_cast<uint64_t>(ordered_key(cand_val[at])) << 32) | static_cast<uint32_t>(~t);
        ++mine;
      }
    }
    s_rank[x] = w;
  }
  if (mine != 0) atomicAdd(&s_valid, mine);
  __syncthreads();
  block_bitonic_sort(s_rank, n2, true);
  const int kk = min(topk, s_valid);
  int k2 = 1;
  while (k2 < kk) k2 <<= 1;
  for (int x = threadIdx.x; x < k2; x += blockDim.x) {
    uint64_t w = ~0ull;  // padding sorts last
    if (x < kk) {
      const uint64_t r = s_rank[x];
      w = (static_cast<uint64_t>(~static_cast<uint32_t>(r)) << 32) | static_cast<uint32_t>(r >> 32);
    }
    s_tok[x] = w;
  }
  __syncthreads();
  if (kk > 1) block_bitonic_sort(s_tok, k2, false);
  int32_t* oi = topk_idx + static_cast<int64_t>(row) * topk;
  float* ov = topk_val != nullptr ? topk_val + static_cast<int64_t>(row) * topk : nullptr;
  for (int x = threadIdx.x; x < topk; x += blockDim.x) {
    if (x < kk) {
      const uint64_t w = s_tok[x];
      oi[x] = static_cast<int32_t>(w >> 32);
      if (ov != nullptr) ov[x] = key_to_float(static_cast<uint32_t>(w));
    } else {
      oi[x] = -1;
      if (ov != nullptr) ov[x] = -__int_as_float(0x7f800000);
    }
  }
}

}  // namespace

// Shared memory of a row's sorts: the candidates rounded up to a power of two, then the kept ones.
size_t merge_candidates_smem(int lists, int k_in) {
  int n2 = 1;
  while (n2 < lists * k_in) n2 <<= 1;
  return sizeof(uint64_t) * (static_cast<size_t>(n2) + kMaxTopk);
}

cudaError_t launch_merge_candidates(const float* cand_val, const int32_t* cand_idx, int lists, int rows, int k_in,
                                    int topk, int32_t* topk_idx, float* topk_val, cudaStream_t stream) {
  cudaError_t e = set_smem_once<merge_candidates_kernel>(merge_candidates_smem(1, IDX_FP4_MERGE_MAX_CANDIDATES));
  if (e != cudaSuccess) return e;
  return launch_pdl(merge_candidates_kernel, dim3(static_cast<unsigned>(rows)), dim3(kMergeThreads),
                    merge_candidates_smem(lists, k_in), stream, 1, false, cand_val, cand_idx, lists, rows, k_in, topk,
                    topk_idx, topk_val);
}

}  // namespace idxfp4
