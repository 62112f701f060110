// MXFP4 tensor-core rate probe: the peak that the prefill scorer's FLOP rate is compared with. The
// kernel issues block-scaled MXFP4 MMAs (tcgen05.mma kind::mxf4, M = 128, N = 128, K = 64: the
// scorers' instruction) back to back from shared-memory operands, so nothing but the tensor pipe
// and the MMA issue limit it. One CTA per SM; eight warps issue (one thread each, as the scorers
// issue from many warps: one issuing thread cannot keep the pipe busy), alternating between two
// accumulators. The operand values do not matter (any E2M1 byte and any finite e8m0 scale is a
// valid input); the accumulators are not read.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace idxfp4 {
namespace {

constexpr int kProbeWarps = 8;
constexpr int kProbeN = 128;
constexpr uint32_t kProbeSmem = 8192 + 8192 + 512 + 512 + 64;  // A, B, their scales, barriers

__global__ void __launch_bounds__(kProbeWarps * 32, 1) mxf4_probe_kernel(int iters, int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tmem_base;
  uint8_t* a = smem;                                      // [4][128][16] E2M1 codes
  uint8_t* b = smem + 8192;                               // [4][128][16]
  uint8_t* sfa = smem + 16384;                            // 512 scale bytes
  uint8_t* sfb = sfa + 512;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sfb + 512);  // [0] scales in TMEM, [1] all MMAs done
  const int tid = static_cast<int>(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < 16384 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0x2A2A2A2Au;
  for (int i = tid; i < 1024 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sfa)[i] = 0x7F7F7F7Fu;  // 2^0
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], kProbeWarps);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t sfa_t = tmem + 2 * kProbeN, sfb_t = sfa_t + 4;
  if (tid == 0) {
    tmem_copy_sf_chunk(sfa_t, smem_addr(sfa));
    tmem_copy_sf_chunk(sfb_t, smem_addr(sfb));
    tc_commit(&bars[0]);
  }
  if (lane == 0) {
    bool ok = mbar_wait(&bars[0], 0, kWaitLimitNs);
    tc_fence_after_sync();
    const uint64_t a_desc = smem_desc(smem_addr(a), 2048, 128);
    const uint64_t b_desc = smem_desc(smem_addr(b), kProbeN * 16, 128);
    const uint32_t idesc0 = mxf4_idesc(128, kProbeN, 0), idesc2 = mxf4_idesc(128, kProbeN, 2);
    const uint32_t d = tmem + static_cast<uint32_t>((warp & 1) * kProbeN);
    if (ok)
#pragma unroll 1
      for (int i = 0; i < iters; ++i) {
        mma_mxf4(d, a_desc, b_desc, idesc0, sfa_t, sfb_t, 1u);
        mma_mxf4(d, a_desc + (4096 >> 4), b_desc + ((2 * kProbeN * 16) >> 4), idesc2, sfa_t, sfb_t, 1u);
      }
    tc_commit(&bars[1]);
    bool done = mbar_wait(&bars[1], 0, kWaitLimitNs);
    if (!ok || !done) set_status(status, IDX_FP4_DEV_TIMEOUT);
    // TMEM is freed only once this warp's MMAs are known to be done (a second bounded wait if not)
    if (!done) done = mbar_wait(&bars[1], 0, kWaitLimitNs);
    (void)done;
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int64_t mxf4_probe_flops(int ctas, int iters) {
  return static_cast<int64_t>(ctas) * kProbeWarps * iters * 2 * (2LL * 128 * kProbeN * 64);
}

cudaError_t launch_mxf4_probe(int ctas, int iters, int32_t* status, cudaStream_t stream) {
  cudaError_t e = set_smem_once<mxf4_probe_kernel>(kProbeSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(mxf4_probe_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kProbeWarps * 32), kProbeSmem, stream,
                    1, false, iters, status);
}

}  // namespace idxfp4
