// decode_g2.cu -- the decode kernels for g = Hq / Hkv = 2 (one translation
// unit per group size, so the variants compile in parallel).
#include "decode_kernels.cuh"

namespace gqa {

cudaError_t launch_decode_group2(const DecodeParams& p, cudaStream_t stream) {
  return launch_group<2>(p, stream);
}

}  // namespace gqa
