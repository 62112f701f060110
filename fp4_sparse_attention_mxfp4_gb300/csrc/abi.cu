// C-ABI entry points: host-side argument checks, then kernel launches on the caller's stream.
// Every check that can fail runs before the first CUDA call, so a rejected call touches
// neither the device nor the stream.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "decode_sched.cuh"
#include "idx_fp4.h"

namespace idxfp4 {
cudaError_t launch_quant_and_cache(const uint16_t* k, int64_t num_tokens, const int32_t* slots, uint8_t* kv_packed,
                                   uint8_t* kv_scale, int64_t num_pages, const uint16_t* q, int64_t num_q_vec,
                                   uint8_t* q_packed, uint8_t* q_scale, int32_t* status, int num_sms,
                                   cudaStream_t stream);
cudaError_t launch_build_decode_schedule(const int32_t* ctx_lens, const int32_t* key_begin, int batch, int next_n,
                                         int max_batch, int64_t max_ctx, int ctas, const DecodeCaps& caps,
                                         void* sched, int32_t* status, cudaStream_t stream);
cudaError_t launch_build_prefill_schedule(const int32_t* cu_seqlens, const int32_t* row_ends, const int32_t* ctx_lens,
                                          int num_requests, int num_rows, int rows_per_unit, int table_width,
                                          int64_t units_cap, int64_t slots_cap, void* workspace, int32_t* status,
                                          cudaStream_t stream);
bool decode_shape_supported(int heads, int next_n);
int64_t mxf4_probe_flops(int ctas, int iters);
cudaError_t launch_mxf4_probe(int ctas, int iters, int32_t* status, cudaStream_t stream);
cudaError_t launch_merge_candidates(const float* cand_val, const int32_t* cand_idx, int lists, int rows, int k_in,
                                    int topk, int32_t* topk_idx, float* topk_val, cudaStream_t stream);
cudaError_t launch_decode(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                          const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                          const int32_t* block_tables, int bt_stride, const int32_t* ctx_lens, int batch, int heads,
                          int next_n, int topk, const void* sched, size_t sched_bytes, void* workspace,
                          size_t ws_bytes, int32_t* topk_idx, float* topk_val, float* logits_debug,
                          int64_t logits_stride, int32_t* status, int grid, cudaStream_t stream);
cudaError_t launch_prefill(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                           const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                           const int32_t* block_tables, int bt_stride, const int32_t* row_ends, int num_rows, int H,
                           int topk, void* workspace, int64_t units_cap, int64_t slots_cap, int32_t* topk_idx,
                           float* topk_val, float* logits_debug, int64_t logits_stride, int32_t* status, int grid,
                           cudaStream_t stream);
}  // namespace idxfp4

namespace {

using namespace idxfp4;

constexpr int64_t kMaxCtx = 1ll << 30;   // keys per sequence / row the sizing formulas accept

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool heads_ok(int h) { return h == 16 || h == 32 || h == 64 || h == 128; }

// Persistent grid: the current device's SM count (capped).
int device_ctas() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms < kMaxCtas ? sms : kMaxCtas;
}

int to_code(cudaError_t e) { return e == cudaSuccess ? IDX_FP4_OK : IDX_FP4_ERR_CUDA; }

// The decode grid: one CTA per SM, at most 256 (a sequence's segment then spans at most 256 CTAs).
int decode_ctas() {
  const int c = device_ctas();
  return c > 256 ? 256 : c;
}

// Decode capacities for (max_batch, max_ctx); false for sizes the tables cannot index (more than
// 2^31 - 1 tiles of 128 keys in all).
bool decode_caps_for(int max_batch, int64_t max_ctx, DecodeCaps* caps) {
  if (max_batch < 1 || max_batch > kMaxBatch || max_ctx < 0 || max_ctx > kMaxCtx) return false;
  *caps = decode_caps(max_batch, max_ctx);
  return caps->tiles_cap <= INT32_MAX && caps->units_cap <= INT32_MAX;
}

size_t decode_ws_bytes(int max_batch, int64_t max_ctx, int topk, int next_n) {
  if (topk < 1 || topk > IDX_FP4_MAX_TOPK || next_n < 1 || next_n > kMaxNextN) return 0;
  DecodeCaps caps;
  if (!decode_caps_for(max_batch, max_ctx, &caps)) return 0;
  return decode_ws_bytes_for(caps, max_batch, next_n, topk);
}

int build_schedule(const int32_t* ctx_lens_dev, const int32_t* key_begin_dev, int batch, int next_n, int max_batch,
                   int64_t max_ctx, void* sched_dev, size_t sched_bytes, int32_t* status_dev, cudaStream_t stream) {
  if (max_batch < 1 || max_batch > kMaxBatch || batch < 0 || batch > max_batch || max_ctx < 0 || max_ctx > kMaxCtx ||
      next_n < 1 || next_n > kMaxNextN)
    return IDX_FP4_ERR_ARG;
  if (sched_dev == nullptr || !aligned16(sched_dev) || (batch > 0 && ctx_lens_dev == nullptr)) return IDX_FP4_ERR_ARG;
  DecodeCaps caps;
  if (!decode_caps_for(max_batch, max_ctx, &caps)) return IDX_FP4_ERR_ARG;
  if (sched_bytes < decode_sched_bytes_for(max_batch, caps)) return IDX_FP4_ERR_CAPACITY;
  const int ctas = decode_ctas();
  if (ctas <= 0) return IDX_FP4_ERR_CUDA;
  return to_code(launch_build_decode_schedule(ctx_lens_dev, key_begin_dev, batch, next_n, max_batch, max_ctx, ctas,
                                              caps, sched_dev, status_dev, stream));
}

int decode_call(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights, const uint8_t* kv_packed,
                const uint8_t* kv_scale, int64_t num_pages, const int32_t* block_tables, int block_table_stride,
                const int32_t* ctx_lens_dev, int batch, int num_heads, int next_n, int topk, const void* sched_dev,
                size_t sched_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx, float* topk_val,
                float* logits_debug, int64_t logits_stride, int32_t* status_dev, cudaStream_t stream) {
  if (!heads_ok(num_heads) || topk < 1 || topk > IDX_FP4_MAX_TOPK || !decode_shape_supported(num_heads, next_n))
    return IDX_FP4_ERR_SHAPE;
  if (batch < 0 || batch > kMaxBatch) return IDX_FP4_ERR_ARG;
  if (batch == 0) return IDX_FP4_OK;
  if (q_packed == nullptr || q_scale == nullptr || weights == nullptr || kv_packed == nullptr ||
      kv_scale == nullptr || block_tables == nullptr || ctx_lens_dev == nullptr || sched_dev == nullptr ||
      workspace == nullptr || topk_idx == nullptr)
    return IDX_FP4_ERR_ARG;
  if (num_pages < 1 || block_table_stride < 1) return IDX_FP4_ERR_ARG;
  if (logits_debug != nullptr && logits_stride < 1) return IDX_FP4_ERR_ARG;
  if (!aligned16(q_packed) || !aligned16(q_scale) || !aligned16(weights) || !aligned16(kv_packed) ||
      !aligned16(kv_scale) || !aligned16(sched_dev) || !aligned16(workspace))
    return IDX_FP4_ERR_ARG;
  if (sched_bytes < sizeof(DecodeSchedHeader)) return IDX_FP4_ERR_CAPACITY;
  const int ctas = decode_ctas();
  if (ctas <= 0) return IDX_FP4_ERR_CUDA;
  return to_code(launch_decode(q_packed, q_scale, weights, kv_packed, kv_scale, num_pages, block_tables,
                               block_table_stride, ctx_lens_dev, batch, num_heads, next_n, topk, sched_dev,
                               sched_bytes, workspace, workspace_bytes, topk_idx, topk_val, logits_debug,
                               logits_stride, status_dev, ctas, stream));
}

}  // namespace

extern "C" {

const char* idx_fp4_error_string(int code) {
  switch (code) {
    case IDX_FP4_OK: return "ok";
    case IDX_FP4_ERR_ARG: return "invalid argument";
    case IDX_FP4_ERR_SHAPE: return "unsupported shape (num_heads must be 16/32/64/128, 1 <= topk <= 2048)";
    case IDX_FP4_ERR_CAPACITY: return "buffer smaller than the sizing function requires";
    case IDX_FP4_ERR_CUDA: return "CUDA launch or device query failed";
    default: return "unknown error code";
  }
}

int idx_fp4_quant_and_cache(const uint16_t* k_bf16, int64_t num_tokens, const int32_t* slot_mapping,
                            uint8_t* kv_packed, uint8_t* kv_scale, int64_t num_pages, const uint16_t* q_bf16,
                            int64_t num_q_rows, int num_heads, uint8_t* q_packed, uint8_t* q_scale,
                            int32_t* status_dev, cudaStream_t stream) {
  if (num_tokens < 0 || num_q_rows < 0 || num_pages < 0) return IDX_FP4_ERR_ARG;
  if (num_tokens > 0) {
    if (k_bf16 == nullptr || slot_mapping == nullptr || kv_packed == nullptr || kv_scale == nullptr)
      return IDX_FP4_ERR_ARG;
    if (!aligned16(k_bf16) || !aligned16(kv_packed)) return IDX_FP4_ERR_ARG;
  }
  int64_t q_vec = 0;
  if (q_bf16 != nullptr && num_q_rows > 0) {
    if (q_packed == nullptr || q_scale == nullptr) return IDX_FP4_ERR_ARG;
    if (!heads_ok(num_heads)) return IDX_FP4_ERR_SHAPE;
    if (!aligned16(q_bf16) || !aligned16(q_packed)) return IDX_FP4_ERR_ARG;
    q_vec = num_q_rows * num_heads;
  }
  if (num_tokens + q_vec == 0) return IDX_FP4_OK;
  const int sms = device_ctas();
  if (sms <= 0) return IDX_FP4_ERR_CUDA;
  return to_code(launch_quant_and_cache(k_bf16, num_tokens, slot_mapping, kv_packed, kv_scale, num_pages, q_bf16,
                                        q_vec, q_packed, q_scale, status_dev, sms, stream));
}

size_t idx_fp4_decode_schedule_bytes(int max_batch, int64_t max_ctx) {
  DecodeCaps caps;
  if (!decode_caps_for(max_batch, max_ctx, &caps)) return 0;
  return decode_sched_bytes_for(max_batch, caps);
}

int idx_fp4_build_decode_schedule(const int32_t* ctx_lens_dev, int batch, int max_batch, int64_t max_ctx,
                                  void* sched_dev, size_t sched_bytes, int32_t* status_dev, cudaStream_t stream) {
  return build_schedule(ctx_lens_dev, nullptr, batch, 1, max_batch, max_ctx, sched_dev, sched_bytes, status_dev,
                        stream);
}

int idx_fp4_build_decode_schedule_range(const int32_t* key_begin_dev, const int32_t* key_end_dev, int batch,
                                        int max_batch, int64_t max_ctx, void* sched_dev, size_t sched_bytes,
                                        int32_t* status_dev, cudaStream_t stream) {
  if (batch > 0 && key_begin_dev == nullptr) return IDX_FP4_ERR_ARG;
  return build_schedule(key_end_dev, key_begin_dev, batch, 1, max_batch, max_ctx, sched_dev, sched_bytes, status_dev,
                        stream);
}

int idx_fp4_build_decode_schedule_mtp(const int32_t* ctx_lens_dev, int batch, int next_n, int max_batch,
                                      int64_t max_ctx, void* sched_dev, size_t sched_bytes, int32_t* status_dev,
                                      cudaStream_t stream) {
  return build_schedule(ctx_lens_dev, nullptr, batch, next_n, max_batch, max_ctx, sched_dev, sched_bytes, status_dev,
                        stream);
}

int64_t idx_fp4_mxf4_probe_flops(int iters) {
  const int ctas = device_ctas();
  if (iters < 1 || ctas <= 0) return 0;
  return mxf4_probe_flops(ctas, iters);
}

int idx_fp4_mxf4_probe(int iters, int32_t* status_dev, cudaStream_t stream) {
  if (iters < 1 || iters > (1 << 20)) return IDX_FP4_ERR_ARG;
  const int ctas = device_ctas();
  if (ctas <= 0) return IDX_FP4_ERR_CUDA;
  return to_code(launch_mxf4_probe(ctas, iters, status_dev, stream));
}

int idx_fp4_merge_candidates(const float* cand_val, const int32_t* cand_idx, int num_lists, int rows, int k_in,
                             int topk, int32_t* topk_idx, float* topk_val, int32_t* status_dev, cudaStream_t stream) {
  (void)status_dev;
  if (num_lists < 1 || rows < 0 || k_in < 1) return IDX_FP4_ERR_ARG;
  if (topk < 1 || topk > IDX_FP4_MAX_TOPK) return IDX_FP4_ERR_SHAPE;
  if (static_cast<int64_t>(num_lists) * k_in > IDX_FP4_MERGE_MAX_CANDIDATES) return IDX_FP4_ERR_CAPACITY;
  if (rows == 0) return IDX_FP4_OK;
  if (cand_val == nullptr || cand_idx == nullptr || topk_idx == nullptr) return IDX_FP4_ERR_ARG;
  return to_code(launch_merge_candidates(cand_val, cand_idx, num_lists, rows, k_in, topk, topk_idx, topk_val, stream));
}

size_t idx_fp4_decode_workspace_bytes(int max_batch, int64_t max_ctx, int topk) {
  return decode_ws_bytes(max_batch, max_ctx, topk, 1);
}

size_t idx_fp4_decode_mtp_workspace_bytes(int max_batch, int64_t max_ctx, int topk, int next_n) {
  return decode_ws_bytes(max_batch, max_ctx, topk, next_n);
}

int idx_fp4_decode_logits_topk(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                               const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                               const int32_t* block_tables, int block_table_stride, const int32_t* ctx_lens_dev,
                               int batch, int num_heads, int topk, const void* sched_dev, size_t sched_bytes,
                               void* workspace, size_t workspace_bytes, int32_t* topk_idx, float* topk_val,
                               float* logits_debug, int64_t logits_stride, int32_t* status_dev,
                               cudaStream_t stream) {
  return decode_call(q_packed, q_scale, weights, kv_packed, kv_scale, num_pages, block_tables, block_table_stride,
                     ctx_lens_dev, batch, num_heads, 1, topk, sched_dev, sched_bytes, workspace, workspace_bytes,
                     topk_idx, topk_val, logits_debug, logits_stride, status_dev, stream);
}

int idx_fp4_decode_mtp_logits_topk(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                                   const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                                   const int32_t* block_tables, int block_table_stride, const int32_t* ctx_lens_dev,
                                   int batch, int next_n, int num_heads, int topk, const void* sched_dev,
                                   size_t sched_bytes, void* workspace, size_t workspace_bytes, int32_t* topk_idx,
                                   float* topk_val, float* logits_debug, int64_t logits_stride, int32_t* status_dev,
                                   cudaStream_t stream) {
  if (next_n < 1 || next_n > kMaxNextN) return IDX_FP4_ERR_SHAPE;
  return decode_call(q_packed, q_scale, weights, kv_packed, kv_scale, num_pages, block_tables, block_table_stride,
                     ctx_lens_dev, batch, num_heads, next_n, topk, sched_dev, sched_bytes, workspace,
                     workspace_bytes, topk_idx, topk_val, logits_debug, logits_stride, status_dev, stream);
}

size_t idx_fp4_prefill_workspace_bytes(int num_requests, int num_rows, int num_heads, int64_t max_ctx, int topk) {
  if (num_requests < 1 || num_requests > kMaxBatch || num_rows < 0 || num_rows > kMaxPrefillRows ||
      !heads_ok(num_heads) || max_ctx < 0 || max_ctx > kMaxCtx || topk < 1 || topk > IDX_FP4_MAX_TOPK)
    return 0;
  return prefill_workspace_bytes_for(num_requests, num_rows, prefill_rows_per_unit(num_heads), max_ctx, topk);
}

int idx_fp4_prefill_logits_topk(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                                const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                                const int32_t* block_tables, int block_table_stride, const int32_t* ctx_lens_dev,
                                const int32_t* cu_seqlens_dev, const int32_t* row_ends_dev, int num_requests,
                                int num_rows, int num_heads, int topk, int64_t max_ctx, void* workspace,
                                size_t workspace_bytes, int32_t* topk_idx, float* topk_val, float* logits_debug,
                                int64_t logits_stride, int32_t* status_dev, cudaStream_t stream) {
  if (!heads_ok(num_heads) || topk < 1 || topk > IDX_FP4_MAX_TOPK) return IDX_FP4_ERR_SHAPE;
  if (num_rows < 0 || num_rows > kMaxPrefillRows || num_requests < 0 || num_requests > kMaxBatch || max_ctx < 0 ||
      max_ctx > kMaxCtx)
    return IDX_FP4_ERR_ARG;
  if (num_rows == 0) return IDX_FP4_OK;
  if (num_requests < 1) return IDX_FP4_ERR_ARG;
  if (q_packed == nullptr || q_scale == nullptr || weights == nullptr || kv_packed == nullptr ||
      kv_scale == nullptr || block_tables == nullptr || ctx_lens_dev == nullptr || cu_seqlens_dev == nullptr ||
      row_ends_dev == nullptr || workspace == nullptr || topk_idx == nullptr)
    return IDX_FP4_ERR_ARG;
  if (num_pages < 1 || block_table_stride < 1) return IDX_FP4_ERR_ARG;
  if (logits_debug != nullptr && logits_stride < 1) return IDX_FP4_ERR_ARG;
  if (!aligned16(q_packed) || !aligned16(q_scale) || !aligned16(weights) || !aligned16(kv_packed) ||
      !aligned16(kv_scale) || !aligned16(workspace))
    return IDX_FP4_ERR_ARG;
  const int q_rows = prefill_rows_per_unit(num_heads);
  if (workspace_bytes < prefill_workspace_bytes_for(num_requests, num_rows, q_rows, max_ctx, topk))
    return IDX_FP4_ERR_CAPACITY;
  const int64_t units_cap = prefill_units_cap(num_requests, num_rows, q_rows, max_ctx);
  const int64_t slots_cap = max_ctx > unit_key_cap(q_rows) ? units_cap * q_rows : 0;
  const int ctas = device_ctas();
  if (ctas <= 0) return IDX_FP4_ERR_CUDA;
  const int grid = static_cast<int>(units_cap < ctas ? units_cap : ctas);
  cudaError_t e = launch_build_prefill_schedule(cu_seqlens_dev, row_ends_dev, ctx_lens_dev, num_requests, num_rows,
                                                q_rows, block_table_stride, units_cap, slots_cap, workspace,
                                                status_dev, stream);
  if (e != cudaSuccess) return IDX_FP4_ERR_CUDA;
  return to_code(launch_prefill(q_packed, q_scale, weights, kv_packed, kv_scale, num_pages, block_tables,
                                block_table_stride, row_ends_dev, num_rows, num_heads, topk, workspace, units_cap,
                                slots_cap, topk_idx, topk_val, logits_debug, logits_stride, status_dev, grid, stream));
}

}  // extern "C"
