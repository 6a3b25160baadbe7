// decode_g8.cu -- the decode kernels for g = Hq / Hkv = 8 (one translation
// unit per group size, so the variants compile in parallel): the per-warp
// MMA kernels of decode_kernels.cuh, whose eight score columns hold the
// eight heads, except with the rotary embedding, whose query takes two
// columns per head: that runs on the tcgen05 kernels of decode_tc.cuh.
#include "decode_tc.cuh"

namespace gqa {

cudaError_t launch_decode_group8(const DecodeParams& p, cudaStream_t stream) {
  if (p.rope_cos != nullptr) return launch_group_tc<8>(p, stream);
  return launch_group<8>(p, stream);
}

}  // namespace gqa
