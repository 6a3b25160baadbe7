// decode.cu -- host side of the split-KV decode (the kernels are in
// decode_kernels.cuh, compiled per group size in decode_g<g>.cu): workspace
// layout, supported sizes, parameter set-up and dispatch, and the
// allocation-free variant's built-in scratch.
#include <cuda.h>

#include <mutex>

#include "decode_params.h"
#include "internal.h"

namespace gqa {

int g_decode_test_skip = -1;
int g_decode_test_cluster = -1;

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

DecodeWorkspace decode_workspace_layout(int B, int Hq, int Hkv, int D) {
  DecodeWorkspace w{};
  const int g = Hq / Hkv;
  w.slots = kDecodeMaxGrid + B * Hkv;
  w.status_off = 0;
  w.ticket_off = 128;
  w.counters_off = 256;
  w.ml_off = align256(w.counters_off + (size_t)B * Hkv * sizeof(uint32_t));
  w.o_off = align256(w.ml_off + (size_t)w.slots * g * 2 * sizeof(float));
  w.total = align256(w.o_off + (size_t)w.slots * g * D * sizeof(float));
  return w;
}

bool decode_supported(int B, int Hq, int Hkv, int L, int D) {
  const int g = Hq / Hkv;
  return D == kDecodeD && (g == 1 || g == 2 || g == 4 || g == 8 || g == 16) && B >= 1 &&
         B <= kDecodeMaxB && L >= 1 && L <= (1 << 24);
}

cudaError_t launch_decode(const void* q, const void* k_new, const void* v_new,
                          const float* rope_cos, const float* rope_sin, bool rope_by_pos,
                          const int32_t* positions, int32_t* advance, const void* k_cache,
                          const void* v_cache, int B, int Hq, int Hkv, int L, int D, int window,
                          float scale, void* out, void* workspace, cudaStream_t stream, int S) {
  const DecodeWorkspace ws = decode_workspace_layout(B, S * Hq, Hkv, D);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  DecodeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.k_new = static_cast<const uint8_t*>(k_new);
  p.v_new = static_cast<const uint8_t*>(v_new);
  p.positions = positions;
  p.k_cache = static_cast<uint8_t*>(const_cast<void*>(k_cache));
  p.v_cache = static_cast<uint8_t*>(const_cast<void*>(v_cache));
  p.out = static_cast<uint16_t*>(out);
  p.status = reinterpret_cast<uint32_t*>(base + ws.status_off);
  p.counters = reinterpret_cast<uint32_t*>(base + ws.counters_off);
  p.part_ml = reinterpret_cast<float*>(base + ws.ml_off);
  p.part_o = reinterpret_cast<float*>(base + ws.o_off);
  p.rope_cos = rope_cos;
  p.rope_sin = rope_sin;
  p.rope_by_pos = rope_by_pos ? 1 : 0;
  p.window = window;
  p.S = S;
  p.test_skip = g_decode_test_skip;
  p.advance = advance;
  p.ticket = reinterpret_cast<uint32_t*>(base + ws.ticket_off);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.L = L;
  p.qscale = scale * 1.4426950408889634f;  // scale * log2(e)
  switch (S * Hq / Hkv) {  // the kernel's heads per KV head: S tokens x g
    case 1: return launch_decode_group1(p, stream);
    case 2: return launch_decode_group2(p, stream);
    case 4: return launch_decode_group4(p, stream);
    case 8: return launch_decode_group8(p, stream);
    case 16: return launch_decode_group16(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gqa

// ---------------------------------------------------------------------------
// attn_decode_step_noalloc: the same decode, with its split-KV scratch in a
// fixed device array instead of a caller-provided workspace, for callers
// that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace gqa {
namespace {

// Upper bound of the built-in scratch; covers every decode size whose
// attn_decode_workspace_size() is at most this (B=256, Hq=64, Hkv=8 needs
// about 12.8 MB).  Every GPU that loads the library keeps this much device
// memory until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The current context's id (0 if none is current or the driver cannot say).
// A device reset (cudaDeviceReset) replaces the context and reloads the
// library's device code, so the array may then sit at another address.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {  // called with the lookup mutex held
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
    resolved = true;
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c ||
      get_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch for the current device.  In host code
// the array's name is only a stand-in, never a usable device address, so the
// address is looked up (cudaGetSymbolAddress, with the device current) once
// per device and context and kept.  The lookup table is guarded by a mutex,
// so host threads making their first calls at the same time are safe; a new
// context on the device (after a reset) triggers a fresh lookup.
void* noalloc_scratch(cudaError_t* err) {
  struct Entry {
    unsigned long long ctx;
    void* addr;
  };
  static std::mutex mu;
  static Entry table[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= 64)) e = cudaErrorInvalidDevice;
  if (e != cudaSuccess) {
    *err = e;
    return nullptr;
  }
  Entry& t = table[dev];
  const unsigned long long ctx = current_context_id();
  if (!t.addr || ctx == 0 || ctx != t.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    // the lookup made the device's context current if none was
    t.ctx = current_context_id();
    t.addr = p;
  }
  *err = cudaSuccess;
  return t.addr;
}

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t launch_decode_noalloc(const void* q, const int32_t* positions, const void* k_cache,
                                  const void* v_cache, int B, int Hq, int Hkv, int L, int D,
                                  float scale, void* out, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  uint8_t* scratch = static_cast<uint8_t*>(noalloc_scratch(&e));
  if (!scratch) return e;
  // The array keeps the previous call's contents: the status word and the
  // arrival counters must start at zero (the partials need no clearing).
  const DecodeWorkspace ws = decode_workspace_layout(B, Hq, Hkv, D);
  e = cudaMemsetAsync(scratch, 0, ws.ml_off, stream);
  if (e != cudaSuccess) return e;
  return launch_decode(q, nullptr, nullptr, nullptr, nullptr, false, positions, nullptr, k_cache,
                       v_cache, B, Hq, Hkv, L, D, 0, scale, out, scratch, stream);
}

}  // namespace gqa
