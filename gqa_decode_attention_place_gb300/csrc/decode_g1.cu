// decode_g1.cu -- the decode kernels for g = Hq / Hkv = 1 (one translation
// unit per group size, so the variants compile in parallel).
#include "decode_kernels.cuh"

namespace gqa {

cudaError_t launch_decode_group1(const DecodeParams& p, cudaStream_t stream) {
  return launch_group<1>(p, stream);
}

}  // namespace gqa
