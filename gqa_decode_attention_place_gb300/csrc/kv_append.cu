// kv_append.cu -- in-place write of one new K row and one new V row per KV head
// into the static cache at each sequence's position ("MiniCPM4 `forward_step`
// Attention Performance Fix", section 4.1: key_cache[:, :, position_id, :] =
// key_states).  A bit-exact 16-byte-vector copy; O(B*Hkv*D) bytes, independent
// of max_len.
#include "common.cuh"
#include "internal.h"

namespace gqa {

// One thread per 16-byte vector of a row; K and V handled by the same thread.
// S rows per sequence (k_new [B, S, Hkv, D]): row t of sequence b goes to
// cache row positions[b] + t.
__global__ void __launch_bounds__(256) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ positions, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int B, int S, int Hkv, int L, int vec_per_row) {
  grid_dependency_wait();
  grid_dependents_launch();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)B * S * Hkv * vec_per_row;
  if (i >= total) return;
  const int c = (int)(i % vec_per_row);
  const long long row = i / vec_per_row;  // (b * S + t) * Hkv + h
  const int h = (int)(row % Hkv);
  const long long bt = row / Hkv;
  const int b = (int)(bt / S), t = (int)(bt % S);
  const int p0 = positions[b];
  if (!rows_in_cache(p0, S - 1, L)) return;  // reported by the decode call
  const long long dst = (((long long)b * Hkv + h) * L + p0 + t) * vec_per_row + c;
  k_cache[dst] = k_new[i];
  v_cache[dst] = v_new[i];
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* positions,
                             void* k_cache, void* v_cache, int B, int Hkv, int L, int D,
                             cudaStream_t stream, int S) {
  const int vec_per_row = D / 8;  // 8 bf16 per 16-byte vector
  const long long total = (long long)B * S * Hkv * vec_per_row;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  return launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                    positions, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), B,
                    S, Hkv, L, vec_per_row);
}

}  // namespace gqa
