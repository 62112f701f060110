// Decode for callers that cannot allocate device memory.
//
// The regular decode call takes a caller-owned workspace for the exchange between the CTAs that
// share a sequence (published histograms, candidate lists, a few counters). Some callers have no way to provide one: code that runs where
// cudaMalloc is not allowed (inside an allocator hook or a custom memory pool that must not
// re-enter itself, in an embedding runtime that owns every device allocation, or on a path
// that must never block on the allocator). For them this file keeps that workspace in a fixed
// array of this library's device memory and calls the regular decode entry point with it.
//
// Cost: kStaticScratchBytes (16 MiB) of device memory on every GPU that loads the library, held
// until the process exits. The array's host-side name is not a device address; its address is
// looked up once per device with cudaGetSymbolAddress while that device is current.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "decode_sched.cuh"
#include "idx_fp4.h"

namespace idxfp4 {
namespace {

constexpr size_t kStaticScratchBytes = IDX_FP4_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Workspace of the decode calls made through idx_fp4_decode_logits_topk_static (zero at load).
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up on first use).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace idxfp4

extern "C" {

size_t idx_fp4_decode_static_bytes(int batch, int64_t max_ctx, int topk) {
  return idx_fp4_decode_workspace_bytes(batch, max_ctx, topk);
}

int idx_fp4_decode_logits_topk_static(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                                      const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                                      const int32_t* block_tables, int block_table_stride,
                                      const int32_t* ctx_lens_dev, int batch, int num_heads, int topk,
                                      int64_t max_ctx, const void* sched_dev, size_t sched_bytes,
                                      int32_t* topk_idx, float* topk_val, float* logits_debug,
                                      int64_t logits_stride, int32_t* status_dev, cudaStream_t stream) {
  using namespace idxfp4;
  if (topk < 1 || topk > IDX_FP4_MAX_TOPK) return IDX_FP4_ERR_SHAPE;
  if (batch < 0 || batch > kMaxBatch || max_ctx < 0 || max_ctx > (int64_t{1} << 30)) return IDX_FP4_ERR_ARG;
  if (batch == 0) return IDX_FP4_OK;
  const size_t need = idx_fp4_decode_static_bytes(batch, max_ctx, topk);
  if (need == 0) return IDX_FP4_ERR_ARG;
  if (need > kStaticScratchBytes) return IDX_FP4_ERR_CAPACITY;
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return IDX_FP4_ERR_CUDA;
  // The layout is the regular call's for a schedule built with (batch, max_ctx). Its
  // synchronisation words must start at zero: a call leaves them at zero, but one that gave up
  // waiting may not, so they are cleared on the stream first (a memset, not an allocation).
  const DecodeCaps caps = decode_caps(batch, max_ctx);
  if (cudaMemsetAsync(scratch, 0, decode_ws_sync_bytes(caps, batch, 1), stream) != cudaSuccess)
    return IDX_FP4_ERR_CUDA;
  return idx_fp4_decode_logits_topk(q_packed, q_scale, weights, kv_packed, kv_scale, num_pages, block_tables,
                                    block_table_stride, ctx_lens_dev, batch, num_heads, topk, sched_dev,
                                    sched_bytes, scratch, need, topk_idx, topk_val, logits_debug, logits_stride,
                                    status_dev, stream);
}

}  // extern "C"
