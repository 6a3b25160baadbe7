// prefill.cu -- causal prefill over a cached prefix (tcgen05 kernel: in progress).
#include "common.cuh"
#include "internal.h"

namespace gqa {

bool prefill_supported(int Hq, int Hkv, int d) { (void)Hq; (void)Hkv; (void)d; return false; }

cudaError_t launch_prefill(const void*, const void*, const void*, int, int, int, int, int, float,
                           void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace gqa
