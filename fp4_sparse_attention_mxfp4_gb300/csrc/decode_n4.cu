// Decode kernel instantiations for 4 query rows per sequence.
#include "decode_kernel.cuh"

namespace idxfp4 {

cudaError_t launch_decode_n4(const DecodeParams& p, int heads, int grid, cudaStream_t stream) {
  switch (heads) {
    case 16: return launch_decode_t<16, 4>(p, grid, stream);
    case 32: return launch_decode_t<32, 4>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idxfp4
