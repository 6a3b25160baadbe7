// internal.h -- launchers behind the C ABI (host side).  Arguments reaching
// these have been validated by capi.cu.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gqa {

// S rows per sequence (k_new [B, S, Hkv, D]) at positions[b] .. + S - 1.
cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* positions,
                             void* k_cache, void* v_cache, int B, int Hkv, int L, int D,
                             cudaStream_t stream, int S = 1);

// Decode workspace layout (bytes), shared by the size query and the launcher.
struct DecodeWorkspace {
  size_t status_off, ticket_off, counters_off, ml_off, o_off, total;
  int slots;
};
DecodeWorkspace decode_workspace_layout(int B, int Hq, int Hkv, int D);

// k_new/v_new null: attention only.  Non-null: the rows are appended at
// positions[b] inside the same launch (kv append fused into decode).
// rope_cos/rope_sin (fp32, only with k_new) non-null: q and the new key row
// are first rotated by the rotary embedding: row b of [B, D] tables, or
// (rope_by_pos) row positions[b] of [L, D] tables.  advance non-null (the
// positions array itself): every position is incremented once the step has
// read them all.  window > 0: attend only rows max(0, pos-window+1)..pos.
// S > 1: multi-token decode (q and out [B, S, Hq, D], token t at
// positions[b] + t; the workspace is laid out for S * Hq heads).
cudaError_t launch_decode(const void* q, const void* k_new, const void* v_new,
                          const float* rope_cos, const float* rope_sin, bool rope_by_pos,
                          const int32_t* positions, int32_t* advance, const void* k_cache,
                          const void* v_cache, int B, int Hq, int Hkv, int L, int D, int window,
                          float scale, void* out, void* workspace, cudaStream_t stream,
                          int S = 1);

// Allocation-free decode: scratch in a fixed device array (decode.cu).
size_t noalloc_scratch_bytes();
cudaError_t launch_decode_noalloc(const void* q, const int32_t* positions, const void* k_cache,
                                  const void* v_cache, int B, int Hq, int Hkv, int L, int D,
                                  float scale, void* out, cudaStream_t stream);

cudaError_t launch_prefill(const void* q, const void* k, const void* v, int S, int start_pos,
                           int Hq, int Hkv, int d, float scale, void* out,
                           cudaStream_t stream);
// Prefill at head dim 64 with one query tile per work item, its keys split
// between the CTA's two softmax warpgroups (prefill_split.cu); maps of
// [tokens, heads, 64] bf16 with a 64 x 1 x 128 box.  scale_log2 = scale *
// log2(e).
cudaError_t launch_prefill_split(const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int S, int start_pos, int Hq, int Hkv,
                                 float scale_log2, void* out, int sms, cudaStream_t stream);
cudaError_t prefill_split_read_timeouts(uint32_t* count);
cudaError_t prefill_split_read_skips(uint32_t* count);
// Prefill waits that gave up since the last call (synchronises the stream).
cudaError_t prefill_read_timeouts(uint32_t* count, cudaStream_t stream);
// Debug builds: prefill accesses a range check skipped since the last call
// (synchronises the stream); 0 in other builds.
cudaError_t prefill_read_skips(uint32_t* count, cudaStream_t stream);

}  // namespace gqa
