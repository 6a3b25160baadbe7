// decode_g4.cu -- the decode kernels for g = Hq / Hkv = 4 (one translation
// unit per group size, so the variants compile in parallel).
#include "decode_kernels.cuh"

namespace gqa {

cudaError_t launch_decode_group4(const DecodeParams& p, cudaStream_t stream) {
  return launch_group<4>(p, stream);
}

}  // namespace gqa
