// Decode entry of the kernel library: the heads x next_n shapes the decode kernel is built for,
// and the dispatch to its instantiations (one translation unit per next_n, built in parallel).
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_kernel.cuh"

namespace idxfp4 {

cudaError_t launch_decode_n1(const DecodeParams& p, int heads, int grid, cudaStream_t stream);
cudaError_t launch_decode_n2(const DecodeParams& p, int heads, int grid, cudaStream_t stream);
cudaError_t launch_decode_n4(const DecodeParams& p, int heads, int grid, cudaStream_t stream);

// Heads and next_n the decode kernel is built for: next_n * heads <= 128.
bool decode_shape_supported(int heads, int next_n) {
  switch (next_n) {
    case 1: return heads == 16 || heads == 32 || heads == 64 || heads == 128;
    case 2: return heads == 16 || heads == 32 || heads == 64;
    case 4: return heads == 16 || heads == 32;
    default: return false;
  }
}

cudaError_t launch_decode(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                          const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                          const int32_t* block_tables, int bt_stride, const int32_t* ctx_lens, int batch, int heads,
                          int next_n, int topk, const void* sched, size_t sched_bytes, void* workspace,
                          size_t ws_bytes, int32_t* topk_idx, float* topk_val, float* logits_debug,
                          int64_t logits_stride, int32_t* status, int grid, cudaStream_t stream) {
  DecodeParams p{};
  p.q_packed = q_packed;
  p.q_scale = q_scale;
  p.weights = weights;
  p.kv_packed = kv_packed;
  p.kv_scale = kv_scale;
  p.num_pages = num_pages;
  p.block_tables = block_tables;
  p.bt_stride = bt_stride;
  p.ctx_lens = ctx_lens;
  p.sched = sched;
  p.sched_bytes = sched_bytes;
  p.batch = batch;
  p.topk = topk;
  p.workspace = workspace;
  p.ws_bytes = ws_bytes;
  p.topk_idx = topk_idx;
  p.topk_val = topk_val;
  p.logits_debug = logits_debug;
  p.logits_stride = logits_stride;
  p.status = status;
  switch (next_n) {
    case 1: return launch_decode_n1(p, heads, grid, stream);
    case 2: return launch_decode_n2(p, heads, grid, stream);
    case 4: return launch_decode_n4(p, heads, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idxfp4
