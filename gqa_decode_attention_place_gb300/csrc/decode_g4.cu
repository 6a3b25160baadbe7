// decode_g4.cu -- the decode kernels for g = Hq / Hkv = 4 (one translation
// unit per group size, so the variants compile in parallel).
#include "decode_tc.cuh"

namespace gqa {

// Few segments (cluster mode): the CUDA-core kernels, whose shorter chain
// of fixed latencies wins at small positions and ties at long ones.  Many
// segments (stream-K): the tensor-core kernels.
cudaError_t launch_decode_group4(const DecodeParams& p, cudaStream_t stream) {
  int C = 0;
  const cudaError_t e = cluster_size<4>(p, &C);
  if (e != cudaSuccess) return e;
  return C > 0 ? launch_group<4>(p, stream) : launch_group_tc<4>(p, stream);
}

}  // namespace gqa
