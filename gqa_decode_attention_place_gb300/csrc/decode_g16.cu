// decode_g16.cu -- the decode kernels for g = Hq / Hkv = 16, or S tokens x g
// query heads = 16 in multi-token decode (one translation unit per group
// size, so the variants compile in parallel).  Tensor cores only: the 16
// heads fill the MMA's N = 16 operand rows.
#include "decode_tc.cuh"

namespace gqa {

cudaError_t launch_decode_group16(const DecodeParams& p, cudaStream_t stream) {
  return launch_group_tc<16>(p, stream);
}

}  // namespace gqa
