// common.cuh -- small sm_103a building blocks shared by the kernels:
// mbarrier pipeline waits with a time limit, bf16 <-> fp32 conversion, the
// ex2 instruction, packed fp32 pairs and the launch with programmatic
// dependent launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "gqa_attn.h"

namespace gqa {

// A pipeline wait that has not completed after this many nanoseconds gives
// up, sets ATTN_DEV_TIMEOUT and lets the kernel return.  A correct launch of
// any supported size waits microseconds at most.
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if the
// wait gave up (time limit) or *abort became non-zero meanwhile.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ------------------------------------------------------------- conversions --

// Two bf16 values packed in a 32-bit word -> two exact fp32 values.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x (the MUFU.EX2 instruction; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch.  wait: block until the kernels this launch
// depends on have completed and their writes are visible (returns at once if
// there are none).  launch: allow the next kernel on the stream to start its
// prologue now.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Packed fp32 pairs (the .f32x2 forms: two IEEE fp32 operations, one issue).
struct f2 {
  unsigned long long r;
};
__device__ __forceinline__ f2 mk2(float lo, float hi) {
  f2 x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x.r) : "f"(lo), "f"(hi));
  return x;
}
__device__ __forceinline__ void brk2(f2 x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x.r));
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.r) : "l"(a.r), "l"(b.r));
  return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.r) : "l"(a.r), "l"(b.r));
  return d;
}

// Whether rows p0 .. p0 + shift (a sequence's position and the shift - 1
// further rows of a multi-token step) lie inside a cache of L rows.  p0 comes
// from the caller and may be any int, so the test is written without a sum
// that could overflow (L >= 1 and 0 <= shift < 2^31 - L keep L - 1 - shift
// in range).
__device__ __forceinline__ bool rows_in_cache(int p0, int shift, int L) {
  return p0 >= 0 && p0 <= L - 1 - shift;
}

__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.r) : "l"(a.r), "l"(b.r), "l"(c.r));
  return d;
}

// Three-input maximum and minimum (one instruction each on sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Debug builds (-DGQA_DEBUG) check the kernels' index-derived accesses:
// tile coordinates of the bulk copies, landing and partial slots, output and
// cache rows.  A failed check sets ATTN_DEV_RANGE in *status (decode) or
// counts in *counter (prefill), and the caller skips the access; nothing
// traps.  Release builds compile every check away.
#ifdef GQA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool range_ok(bool ok, uint32_t* status) {
  if (!kDebugChecks || ok) return true;
  set_status(status, ATTN_DEV_RANGE);
  return false;
}
__device__ __forceinline__ bool range_ok_count(bool ok, unsigned int* counter) {
  if (!kDebugChecks || ok) return true;
  atomicAdd(counter, 1u);
  return false;
}

// Launch `kernel` on `stream` with programmatic stream serialisation, so it
// may begin while the previous kernel on the stream drains (the kernel calls
// grid_dependency_wait() before touching anything that kernel wrote).
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace gqa
