// decode_g8.cu -- the decode kernels for g = Hq / Hkv = 8 (one translation
// unit per group size, so the variants compile in parallel).
#include "decode_tc.cuh"

namespace gqa {

cudaError_t launch_decode_group8(const DecodeParams& p, cudaStream_t stream) {
  return launch_group_tc<8>(p, stream);
}

}  // namespace gqa
