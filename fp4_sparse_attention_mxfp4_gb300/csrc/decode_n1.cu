// Decode kernel instantiations for 1 query row per sequence.
#include "decode_kernel.cuh"

namespace idxfp4 {

cudaError_t launch_decode_n1(const DecodeParams& p, int heads, int grid, cudaStream_t stream) {
  switch (heads) {
    case 16: return launch_decode_t<16, 1>(p, grid, stream);
    case 32: return launch_decode_t<32, 1>(p, grid, stream);
    case 64: return launch_decode_t<64, 1>(p, grid, stream);
    case 128: return launch_decode_t<128, 1>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idxfp4
