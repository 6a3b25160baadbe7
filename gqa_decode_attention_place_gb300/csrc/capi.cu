// capi.cu -- the extern "C" entry points declared in include/gqa_attn.h:
// argument validation on the host, then one launch on the caller's stream.
#include <cstdint>

#include "gqa_attn.h"
#include "decode_params.h"
#include "internal.h"

namespace gqa {
bool decode_supported(int B, int Hq, int Hkv, int L, int D);
bool prefill_supported(int Hq, int Hkv, int d);
}  // namespace gqa

namespace {

thread_local int g_last_cuda_error = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  g_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int attn_kv_append(const void* k_new, const void* v_new, const int32_t* positions,
                   void* k_cache, void* v_cache, int B, int Hkv, int L, int D,
                   cudaStream_t stream) {
  if (!k_new || !v_new || !positions || !k_cache || !v_cache) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hkv <= 0 || L <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (D % 8 != 0 || D > 256) return ATTN_ERR_UNSUPPORTED;
  return cuda_status(
      gqa::launch_kv_append(k_new, v_new, positions, k_cache, v_cache, B, Hkv, L, D, stream));
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int L, int D) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || D <= 0 || Hq % Hkv != 0) return 0;
  if (!gqa::decode_supported(B, Hq, Hkv, L, D)) return 0;
  return gqa::decode_workspace_layout(B, Hq, Hkv, D).total;
}

int attn_decode_step(const void* q, const int32_t* positions, const void* k_cache,
                     const void* v_cache, int B, int Hq, int Hkv, int L, int D, float scale,
                     void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !positions || !k_cache || !v_cache || !out) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || D <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (!gqa::decode_supported(B, Hq, Hkv, L, D)) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < gqa::decode_workspace_layout(B, Hq, Hkv, D).total)
    return ATTN_ERR_WORKSPACE;
  return cuda_status(gqa::launch_decode(q, nullptr, nullptr, nullptr, nullptr, false, positions,
                                        nullptr, k_cache, v_cache, B, Hq, Hkv, L, D, 0, scale, out,
                                        workspace, stream));
}

namespace {

int decode_append(const void* q, const void* k_new, const void* v_new, const float* rope_cos,
                  const float* rope_sin, bool rope_by_pos, const int32_t* positions,
                  int32_t* advance, void* k_cache, void* v_cache, int B, int Hq, int Hkv, int L,
                  int D, float scale, void* out, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream, int window = 0) {
  if (!q || !positions || !k_cache || !v_cache || !out || !k_new != !v_new)
    return ATTN_ERR_INVALID_ARG;
  if (!k_new && (rope_cos || advance)) return ATTN_ERR_INVALID_ARG;
  if (window < 0) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || D <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || (k_new && (!aligned16(k_new) || !aligned16(v_new))) ||
      !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (!gqa::decode_supported(B, Hq, Hkv, L, D)) return ATTN_ERR_UNSUPPORTED;
  // the rotated query takes two operand rows per head (bf16 high and low
  // parts) in the tensor-core kernels' 16 rows: g <= 8 with the rotation
  if (rope_cos && Hq / Hkv > 8) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < gqa::decode_workspace_layout(B, Hq, Hkv, D).total)
    return ATTN_ERR_WORKSPACE;
  return cuda_status(gqa::launch_decode(q, k_new, v_new, rope_cos, rope_sin, rope_by_pos,
                                        positions, advance, k_cache, v_cache, B, Hq, Hkv, L, D,
                                        window, scale, out, workspace, stream));
}

}  // namespace

int attn_decode_step_append(const void* q, const void* k_new, const void* v_new,
                            const int32_t* positions, void* k_cache, void* v_cache, int B,
                            int Hq, int Hkv, int L, int D, float scale, void* out,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!k_new || !v_new) return ATTN_ERR_INVALID_ARG;
  return decode_append(q, k_new, v_new, nullptr, nullptr, false, positions, nullptr, k_cache,
                       v_cache, B, Hq, Hkv, L, D, scale, out, workspace, workspace_bytes, stream);
}

int attn_decode_step_rope_append(const void* q, const void* k_new, const void* v_new,
                                 const float* cos, const float* sin, const int32_t* positions,
                                 void* k_cache, void* v_cache, int B, int Hq, int Hkv, int L,
                                 int D, float scale, void* out, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  if (!k_new || !v_new) return ATTN_ERR_INVALID_ARG;
  if (!cos || !sin || !aligned16(cos) || !aligned16(sin)) return ATTN_ERR_INVALID_ARG;
  return decode_append(q, k_new, v_new, cos, sin, false, positions, nullptr, k_cache, v_cache, B,
                       Hq, Hkv, L, D, scale, out, workspace, workspace_bytes, stream);
}

int attn_decode_step_window(const void* q, const void* k_new, const void* v_new,
                            const int32_t* positions, void* k_cache, void* v_cache, int B, int Hq,
                            int Hkv, int L, int D, int window, float scale, void* out,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (window <= 0) return ATTN_ERR_INVALID_ARG;
  return decode_append(q, k_new, v_new, nullptr, nullptr, false, positions, nullptr, k_cache,
                       v_cache, B, Hq, Hkv, L, D, scale, out, workspace, workspace_bytes, stream,
                       window);
}

int attn_decode_multi(const void* q, const void* k_new, const void* v_new,
                      const int32_t* positions, void* k_cache, void* v_cache, int B, int S,
                      int Hq, int Hkv, int L, int D, float scale, void* out, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !positions || !k_cache || !v_cache || !out || !k_new != !v_new)
    return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || D <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || (k_new && (!aligned16(k_new) || !aligned16(v_new))) ||
      !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if ((long long)S * Hq > 65536 || !gqa::decode_supported(B, S * Hq, Hkv, L, D))
    return ATTN_ERR_UNSUPPORTED;  // S * g must be 1, 2, 4, 8 or 16
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < gqa::decode_workspace_layout(B, S * Hq, Hkv, D).total)
    return ATTN_ERR_WORKSPACE;
  if (k_new) {
    const int st = cuda_status(gqa::launch_kv_append(k_new, v_new, positions, k_cache, v_cache, B,
                                                     Hkv, L, D, stream, S));
    if (st != ATTN_OK) return st;
  }
  return cuda_status(gqa::launch_decode(q, nullptr, nullptr, nullptr, nullptr, false, positions,
                                        nullptr, k_cache, v_cache, B, Hq, Hkv, L, D, 0, scale,
                                        out, workspace, stream, S));
}

int attn_decode_stream_step(const void* q, const void* k_new, const void* v_new,
                            const float* cos_table, const float* sin_table, int32_t* positions,
                            void* k_cache, void* v_cache, int B, int Hq, int Hkv, int L, int D,
                            float scale, void* out, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  if (!k_new || !v_new) return ATTN_ERR_INVALID_ARG;
  if ((cos_table == nullptr) != (sin_table == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (cos_table && (!aligned16(cos_table) || !aligned16(sin_table))) return ATTN_ERR_INVALID_ARG;
  return decode_append(q, k_new, v_new, cos_table, sin_table, true, positions, positions, k_cache,
                       v_cache, B, Hq, Hkv, L, D, scale, out, workspace, workspace_bytes, stream);
}

int attn_decode_step_noalloc(const void* q, const int32_t* positions, const void* k_cache,
                             const void* v_cache, int B, int Hq, int Hkv, int L, int D,
                             float scale, void* out, cudaStream_t stream) {
  if (!q || !positions || !k_cache || !v_cache || !out) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || D <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (!gqa::decode_supported(B, Hq, Hkv, L, D)) return ATTN_ERR_UNSUPPORTED;
  if (gqa::decode_workspace_layout(B, Hq, Hkv, D).total > gqa::noalloc_scratch_bytes())
    return ATTN_ERR_WORKSPACE;  // beyond the built-in scratch
  return cuda_status(gqa::launch_decode_noalloc(q, positions, k_cache, v_cache, B, Hq, Hkv, L,
                                                D, scale, out, stream));
}

int attn_prefill_causal(const void* q, const void* k, const void* v, int S, int start_pos,
                        int Hq, int Hkv, int d, float scale, void* out, cudaStream_t stream) {
  if (S < 0 || start_pos < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((long long)start_pos + S >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  if (!gqa::prefill_supported(Hq, Hkv, d)) return ATTN_ERR_UNSUPPORTED;
  if (S == 0) return ATTN_OK;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return ATTN_ERR_INVALID_ARG;
  return cuda_status(
      gqa::launch_prefill(q, k, v, S, start_pos, Hq, Hkv, d, scale, out, stream));
}

int attn_read_prefill_status(uint32_t* timeouts, cudaStream_t stream) {
  uint32_t n = 0;
  const cudaError_t e = gqa::prefill_read_timeouts(&n, stream);
  if (e != cudaSuccess) return cuda_status(e);
  if (timeouts) *timeouts = n;
  return n ? ATTN_ERR_DEVICE : ATTN_OK;
}

int attn_read_prefill_skips(uint32_t* skips, cudaStream_t stream) {
  uint32_t n = 0;
  const cudaError_t e = gqa::prefill_read_skips(&n, stream);
  if (e != cudaSuccess) return cuda_status(e);
  if (skips) *skips = n;
  return n ? ATTN_ERR_DEVICE : ATTN_OK;
}

int attn_debug_build(void) {
#ifdef GQA_DEBUG
  return 1;
#else
  return 0;
#endif
}

int attn_read_device_status(void* workspace, uint32_t* bits, cudaStream_t stream) {
  if (!workspace) return ATTN_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(workspace, 0, sizeof(word));
  if (e != cudaSuccess) return cuda_status(e);
  if (bits) *bits = word;
  return word ? ATTN_ERR_DEVICE : ATTN_OK;
}

int attn_test_force_schedule(int cluster) {
  if (cluster < -1 || cluster > 16) return ATTN_ERR_INVALID_ARG;
  gqa::g_decode_test_cluster = cluster;
  return ATTN_OK;
}

int attn_test_skip_tile(int tile) {
  if (tile < -1) return ATTN_ERR_INVALID_ARG;
  gqa::g_decode_test_skip = tile;
  return ATTN_OK;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported size";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE: return "device flagged an error";
    default: return "unknown status";
  }
}

int attn_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
