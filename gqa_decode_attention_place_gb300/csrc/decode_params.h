// decode_params.h -- the decode kernels' launch parameters and the sizes the
// host-side code (workspace layout, argument checks) shares with them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gqa {

constexpr int kDecodeD = 128;         // head dim of the decode kernels
constexpr int kDecodeMaxB = 8192;     // sequences per launch
constexpr int kDecodeMaxGrid = 1024;  // stream-K CTAs (workspace partial slots)

struct DecodeParams {
  const uint16_t* q;
  const uint8_t* k_new;  // [B, Hkv, D] rows to append at positions[b], or null
  const uint8_t* v_new;
  const int32_t* positions;
  uint8_t* k_cache;  // written only by the fused append (row positions[b])
  uint8_t* v_cache;
  uint16_t* out;
  uint32_t* status;
  uint32_t* counters;
  float* part_ml;
  float* part_o;
  const float* rope_cos;  // rotation (with k_new), or null: [B, D] rows, or a
  const float* rope_sin;  // [L, D] table indexed by position (rope_by_pos)
  int32_t* advance;       // the positions array, to add 1 to after the step, or null
  uint32_t* ticket;       // grid-wide arrival counter for the advance
  int rope_by_pos;
  int window;             // 0: rows 0..pos; W > 0: rows max(0, pos-W+1)..pos
  int S;                  // new tokens per sequence (1; > 1: multi-token decode)
  int test_skip;          // failure-path tests: a tile never issued, or -1
  int B, Hq, Hkv, L;
  float qscale;  // scale * log2(e)
};

// Failure-path tests: a tile of the first segment the next decode launches
// will not issue (-1: none).  Process-wide; set through attn_test_skip_tile.
extern int g_decode_test_skip;
// Schedule tests: -1 chooses the split of each segment automatically; 0
// forces stream-K; C >= 1 forces cluster mode with clusters of C CTAs.
// Process-wide; set through attn_test_force_schedule.
extern int g_decode_test_cluster;

// One launcher per group size g = Hq / Hkv (decode_g<g>.cu).
cudaError_t launch_decode_group1(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_group2(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_group4(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_group8(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_group16(const DecodeParams& p, cudaStream_t stream);

}  // namespace gqa
