// Writer: bf16 keys -> MXFP4 in the paged two-plane cache; bf16 query heads -> plain MXFP4.
//
// "Score a DSA sparse indexer in FP4" (squashed commit message: the FP4 output mode of the
// fused writer stores packed E2M1 plus e8m0 scales in the index region; sub-commit
// "Schedule, refuse and document ...": rows with slot < 0 are skipped). One warp encodes one
// 128-dim vector: lane l owns dims 4l..4l+3, the 8 lanes of a 32-dim group reduce the
// group's max magnitude with shuffles, and each lane stores its two packed bytes. With enough
// vectors to fill the GPU a warp takes four consecutive vectors at a time and issues their loads
// together; a small input (a decode step's few keys and queries) keeps one vector per warp and
// spreads over more SMs.
// HBM-bound: 256 B read and 68 B written per vector.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace idxfp4 {
namespace {

// e = the smallest integer with amax <= 6 * 2^e, clamped to [-127, 127], from the bits of a
// non-negative finite float: amax = m * 2^E with m in [1, 2) gives e = E - 2 when m <= 1.5 and
// E - 1 otherwise. Subnormal or zero amax lands at the clamp.
__device__ __forceinline__ int block_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>(b >> 23);
  if (ef == 0) return -127;
  const int e = (ef - 127) - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Nearest E2M1 magnitude code of a >= 0 (already divided by the scale), ties to the even code.
__device__ __forceinline__ uint32_t e2m1_code(float a) {
  return static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) + static_cast<uint32_t>(a > 1.25f) +
         static_cast<uint32_t>(a >= 1.75f) + static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
         static_cast<uint32_t>(a > 5.0f);
}

__device__ __forceinline__ float bf16_lo(uint32_t two) { return __uint_as_float(two << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t two) { return __uint_as_float(two & 0xFFFF0000u); }

// Encode the warp's vector from this lane's dims 4l..4l+3 (raw bf16 pairs). Returns this lane's 2
// packed bytes and the group's scale byte (valid in every lane).
__device__ __forceinline__ void encode_lane(uint2 raw, uint32_t& packed2, uint32_t& scale_byte) {
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
  const int e = block_exponent(amax);
  // 2^-e exactly: a normal float for e <= 126, the subnormal 2^-127 for e = 127.
  const float inv = (127 - e) > 0 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(0x00400000u);
  uint32_t out = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float y = __fmul_rn(fabsf(x[j]), inv);
    const uint32_t code = e2m1_code(y) | (x[j] < 0.0f ? 8u : 0u);
    out |= code << (4 * j);
  }
  packed2 = out;
  scale_byte = static_cast<uint32_t>(e + 127);
}

template <int kVecPerWarp>
__global__ void __launch_bounds__(256) quant_and_cache_kernel(const uint16_t* __restrict__ k, int64_t num_tokens,
                                                              const int32_t* __restrict__ slots, uint8_t* kv_packed,
                                                              uint8_t* kv_scale, int64_t num_pages,
                                                              const uint16_t* __restrict__ q, int64_t num_q_vec,
                                                              uint8_t* q_packed, uint8_t* q_scale, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int g = lane >> 3;        // 32-dim group of this lane
  const int byte_in_group = (lane & 7) * 2;
  const int64_t total = num_tokens + num_q_vec;
  for (int64_t v0 = warp * kVecPerWarp; v0 < total; v0 += nwarps * kVecPerWarp) {
    uint2 raw[kVecPerWarp];
    int64_t slot[kVecPerWarp];
#pragma unroll
    for (int i = 0; i < kVecPerWarp; ++i) {
      const int64_t v = v0 + i;
      raw[i] = make_uint2(0u, 0u);
      slot[i] = -1;
      if (v < num_tokens) slot[i] = slots[v];
      if (v < total)
        raw[i] = __ldg(reinterpret_cast<const uint2*>(v < num_tokens ? k + v * kHeadDim : q + (v - num_tokens) * kHeadDim) +
                       lane);
    }
#pragma unroll
    for (int i = 0; i < kVecPerWarp; ++i) {
      const int64_t v = v0 + i;
      if (v >= total) break;
      if (v < num_tokens) {
        if (slot[i] < 0) continue;
        if (slot[i] >= num_pages * kPage) {
          if (lane == 0) set_status(status, IDX_FP4_DEV_BAD_SLOT);
          continue;
        }
        uint32_t packed2, sb;
        encode_lane(raw[i], packed2, sb);
        const int64_t page = slot[i] / kPage;
        const int row = static_cast<int>(slot[i] % kPage);
        uint8_t* dst = kv_packed + page * kPageBytes + (static_cast<int64_t>(g) * kPage + row) * 16 + byte_in_group;
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed2);
        if ((lane & 7) == 0) kv_scale[page * kPageScaleBytes + g * kPage + scale_slot(row)] = static_cast<uint8_t>(sb);
      } else {
        const int64_t qv = v - num_tokens;
        uint32_t packed2, sb;
        encode_lane(raw[i], packed2, sb);
        *reinterpret_cast<uint16_t*>(q_packed + qv * 64 + g * 16 + byte_in_group) = static_cast<uint16_t>(packed2);
        if ((lane & 7) == 0) q_scale[qv * 4 + g] = static_cast<uint8_t>(sb);
      }
    }
  }
}

}  // namespace

cudaError_t launch_quant_and_cache(const uint16_t* k, int64_t num_tokens, const int32_t* slots, uint8_t* kv_packed,
                                   uint8_t* kv_scale, int64_t num_pages, const uint16_t* q, int64_t num_q_vec,
                                   uint8_t* q_packed, uint8_t* q_scale, int32_t* status, int num_sms,
                                   cudaStream_t stream) {
  const int64_t vecs = num_tokens + num_q_vec;
  if (vecs == 0) return cudaSuccess;
  // four vectors per warp once that still gives every SM four blocks of 8 warps
  const bool wide = vecs >= static_cast<int64_t>(num_sms) * 4 * 8 * 4;
  const int per_block = wide ? 8 * 4 : 8;
  const int64_t blocks_needed = (vecs + per_block - 1) / per_block;
  const int blocks = static_cast<int>(blocks_needed < static_cast<int64_t>(num_sms) * 16 ? blocks_needed
                                                                                          : static_cast<int64_t>(num_sms) * 16);
  if (wide)
    return launch_pdl(quant_and_cache_kernel<4>, dim3(blocks), dim3(256), 0, stream, 1, false, k, num_tokens, slots,
                      kv_packed, kv_scale, num_pages, q, num_q_vec, q_packed, q_scale, status);
  return launch_pdl(quant_and_cache_kernel<1>, dim3(blocks), dim3(256), 0, stream, 1, false, k, num_tokens, slots,
                    kv_packed, kv_scale, num_pages, q, num_q_vec, q_packed, q_scale, status);
}

}  // namespace idxfp4
