// prefill.cu -- causal prefill over a cached prefix on the tcgen05 tensor cores.
//
// What it computes ("step14_3 -- batched attention", sections "problem" and
// "F.scaled_dot_product_attention"; "MiniCPM4 `forward_step` Attention
// Performance Fix", section 5: batch prefill is causal): S new tokens at
// absolute positions start_pos..start_pos+S-1, q [S,Hq,d], k/v
// [start_pos+S,Hkv,d] (prefix rows first); token i attends keys
// 0..start_pos+i (causal mask aligned to the bottom-right corner), query head
// h reads KV head h/g.  out [S,Hq,d] bf16.
//
// How (one CTA per (128-token query tile, query head); longest tiles first):
//  * warp 0, one thread: TMA (cp.async.bulk.tensor, 128-byte swizzle) loads the
//    Q tile once and streams 128-key K and V tiles through a 2-stage ring.
//  * warp 1, one thread: issues tcgen05.mma (bf16 in, fp32 accumulate in
//    tensor memory): S = Q K^T into 128 TMEM columns, then O_tile = P V into
//    one of two 64-column TMEM buffers.  S of tile i+1 is issued as soon as
//    the softmax has read S of tile i, so QK^T overlaps the softmax.
//  * warps 4-7 (128 threads, thread r owns query row r): read the S row from
//    TMEM, mask the causal diagonal, keep the online softmax (running max and
//    sum in base 2), write P as bf16 into shared memory in the 128-byte
//    swizzled K-major layout the MMA reads, and fold each finished O_tile into
//    a register accumulator: O = O * exp2(m_old - m_new) + O_tile.
//  Scores never leave the SM (no S or P in HBM).
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

constexpr int kBM = 128;   // query rows per CTA (MMA M)
constexpr int kBN = 128;   // keys per tile (MMA N of QK^T, K of PV)
constexpr int kHD = 64;    // head dim (MMA K of QK^T, N of PV)
constexpr int kKVStages = 2;
constexpr int kPThreads = 256;
constexpr int kTileBytes = kBM * kHD * 2;  // 16 KB: a 128 x 64 bf16 tile
constexpr uint32_t kTmemCols = 256;        // S: 128, O_tile x2: 2 x 64

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kTileBytes;                     // stage s: K, then V
constexpr int kOffP = kOffKV + kKVStages * 2 * kTileBytes;     // P: keys 0-63, 64-127
constexpr int kOffBar = kOffP + 2 * kTileBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;               // + alignment slack

// barrier slots
constexpr int kBarQ = 0;
constexpr int kBarKVFull = 1;                 // + stage
constexpr int kBarKVEmpty = kBarKVFull + kKVStages;
constexpr int kBarSFull = kBarKVEmpty + kKVStages;
constexpr int kBarSFree = kBarSFull + 1;
constexpr int kBarPFull = kBarSFree + 1;
constexpr int kBarPVDone = kBarPFull + 1;     // + buffer (2)
constexpr int kNumBars = kBarPVDone + 2;

__device__ unsigned int g_prefill_timeouts;   // diagnostic: waits that gave up

struct PrefillParams {
  uint16_t* out;
  int S, start_pos, Hq, Hkv, g, n_qt;
  float scale_log2;  // scale * log2(e)
};

// ---------------------------------------------------------- PTX wrappers --

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a tcgen05 operand in the 128-byte
// swizzled canonical layout (8-row x 128-byte swizzle atoms, atoms 1024 bytes
// apart along the strided dimension).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4)                       // D = f32
         | (1u << 7)                     // A = bf16
         | (1u << 10)                    // B = bf16
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_wait(bar, parity, abort_flag)) return true;
  if (!*abort_flag) atomicAdd(&g_prefill_timeouts, 1u);
  *abort_flag = 1;
  return false;
}

__global__ void __launch_bounds__(kPThreads, 1)
    prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.Hq;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x / p.Hq);  // longest (last) tiles first
  const int q0 = qt * kBM;
  const int kvh = h / p.g;
  const int q_last = min(q0 + kBM, p.S);              // one past the last valid row
  const int n_tiles = (p.start_pos + q_last + kBN - 1) / kBN;

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(bar(kBarKVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 128);
    mbar_init(bar(kBarPFull), 128);
    mbar_init(bar(kBarPVDone + 0), 1);
    mbar_init(bar(kBarPVDone + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tm_S = tmem;            // columns [0, 128)
  const uint32_t tm_O0 = tmem + 128;     // columns [128, 192)
  const uint32_t sQ = base + kOffQ;
  const uint32_t sP = base + kOffP;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(kBarQ), kTileBytes);
      tma_load_3d(sQ, &tm_q, 0, h, q0, bar(kBarQ));
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kKVStages;
        const uint32_t u = (uint32_t)(i / kKVStages);
        if (i >= kKVStages && !wait_or_abort(bar(kBarKVEmpty + s), (u - 1) & 1u, abort_flag)) break;
        const uint32_t sK = base + kOffKV + s * 2 * kTileBytes;
        mbar_arrive_expect_tx(bar(kBarKVFull + s), 2 * kTileBytes);
        tma_load_3d(sK, &tm_k, 0, kvh, i * kBN, bar(kBarKVFull + s));
        tma_load_3d(sK + kTileBytes, &tm_v, 0, kvh, i * kBN, bar(kBarKVFull + s));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(kBM, kBN, false);
      constexpr uint32_t idesc_pv = make_idesc(kBM, kHD, true);
      auto issue_s = [&](int i) -> bool {
        const int s = i % kKVStages;
        if (!wait_or_abort(bar(kBarKVFull + s), (uint32_t)(i / kKVStages) & 1u, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t sK = base + kOffKV + s * 2 * kTileBytes;
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k)
          tc_mma(tm_S, sw128_desc(sQ + k * 32), sw128_desc(sK + k * 32), idesc_qk, k > 0);
        tc_commit(bar(kBarSFull));
        return true;
      };
      bool ok = wait_or_abort(bar(kBarQ), 0, abort_flag) && issue_s(0);
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (i + 1 < n_tiles) {
          // the softmax has read S_i: issue S_{i+1} while it works on tile i
          ok = wait_or_abort(bar(kBarSFree), (uint32_t)i & 1u, abort_flag) && issue_s(i + 1);
          if (!ok) break;
        }
        if (!wait_or_abort(bar(kBarPFull), (uint32_t)i & 1u, abort_flag)) break;
        tc_fence_after();
        const int s = i % kKVStages;
        const uint32_t sV = base + kOffKV + s * 2 * kTileBytes + kTileBytes;
        const uint32_t tm_O = tm_O0 + (uint32_t)(i & 1) * kHD;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          tc_mma(tm_O, sw128_desc(sP + (k >> 2) * kTileBytes + (k & 3) * 32),
                 sw128_desc(sV + k * 16 * 128), idesc_pv, k > 0);
        tc_commit(bar(kBarPVDone + (i & 1)));
        tc_commit(bar(kBarKVEmpty + s));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------- softmax / epilogue (r) --
    const int r = (warp - 4) * 32 + lane;              // query row of this thread
    const uint32_t lane_off = (uint32_t)((warp - 4) * 32) << 16;
    const int qpos = p.start_pos + q0 + r;             // absolute position of the row
    float m_run = -INFINITY, l_run = 0.f, alpha_prev = 0.f;
    float o[kHD];
#pragma unroll
    for (int j = 0; j < kHD; ++j) o[j] = 0.f;

    auto fold = [&](int i) -> bool {  // o = o * alpha_prev + O_tile_i
      if (!wait_or_abort(bar(kBarPVDone + (i & 1)), (uint32_t)(i >> 1) & 1u, abort_flag))
        return false;
      tc_fence_after();
      const uint32_t tm_O = tm_O0 + (uint32_t)(i & 1) * kHD + lane_off;
      float t0[32], t1[32];
      tmem_ld32(tm_O, t0);
      tmem_ld32(tm_O + 32, t1);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        o[j] = fmaf(o[j], alpha_prev, t0[j]);
        o[32 + j] = fmaf(o[32 + j], alpha_prev, t1[j]);
      }
      return true;
    };

    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      if (!wait_or_abort(bar(kBarSFull), (uint32_t)i & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float sv[kBN];
      {
        float c[32];
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          tmem_ld32(tm_S + lane_off + cc * 32, c);
#pragma unroll
          for (int j = 0; j < 32; ++j) sv[cc * 32 + j] = c[j];
        }
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarSFree));

      // causal mask (only tiles reaching past this row's position) and max
      const int kbase = i * kBN;
      float mx = -INFINITY;
      if (kbase + kBN - 1 > qpos) {
#pragma unroll
        for (int j = 0; j < kBN; ++j) {
          sv[j] = (kbase + j <= qpos) ? sv[j] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sv[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kBN; ++j) {
          sv[j] *= p.scale_log2;
          mx = fmaxf(mx, sv[j]);
        }
      }
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m_run - m_use);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < kBN; ++j) {
        sv[j] = ex2(sv[j] - m_use);
        rs += sv[j];
      }
      l_run = l_run * alpha + rs;
      m_run = m_new;

      // PV_{i-1} finished: fold it, and P's buffer is free again
      if (i > 0 && !fold(i - 1)) { ok = false; break; }

      // P row r -> shared memory, 128-byte swizzle: 16-byte chunk c of row r
      // sits at chunk position c ^ (r % 8); keys 0-63 and 64-127 in two tiles
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        const uint32_t w0 = pack_bf16x2(sv[c * 8 + 0], sv[c * 8 + 1]);
        const uint32_t w1 = pack_bf16x2(sv[c * 8 + 2], sv[c * 8 + 3]);
        const uint32_t w2 = pack_bf16x2(sv[c * 8 + 4], sv[c * 8 + 5]);
        const uint32_t w3 = pack_bf16x2(sv[c * 8 + 6], sv[c * 8 + 7]);
        const uint32_t addr =
            sP + (c >> 3) * kTileBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1),
                     "r"(w2), "r"(w3)
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
      alpha_prev = alpha;
    }
    if (ok) ok = fold(n_tiles - 1);

    // epilogue: normalise and store row r (128 contiguous bytes)
    if (q0 + r < p.S) {
      const float inv = ok ? 1.f / l_run : __int_as_float(0x7fc00000);
      uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)(q0 + r) * p.Hq + h) * kHD);
#pragma unroll
      for (int c = 0; c < kHD / 8; ++c) {
        uint4 v;
        v.x = pack_bf16x2(o[c * 8 + 0] * inv, o[c * 8 + 1] * inv);
        v.y = pack_bf16x2(o[c * 8 + 2] * inv, o[c * 8 + 3] * inv);
        v.z = pack_bf16x2(o[c * 8 + 4] * inv, o[c * 8 + 5] * inv);
        v.w = pack_bf16x2(o[c * 8 + 6] * inv, o[c * 8 + 7] * inv);
        dst[c] = v;
      }
    }
  }

  // ------------------------------------------------------------ teardown --
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let tensor-core work and copies still in flight land before freeing TMEM
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// [tokens, heads, 64] bf16 viewed as 3-D (64, heads, tokens); box 64 x 1 x 128.
bool make_map(CUtensorMap* m, const void* ptr, int tokens, int heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHD, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)kHD * 2, (cuuint64_t)heads * kHD * 2};
  cuuint32_t box[3] = {(cuuint32_t)kHD, 1, (cuuint32_t)kBM};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int Hq, int Hkv, int d) {
  return d == kHD && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && Hq <= 65535;
}

cudaError_t launch_prefill(const void* q, const void* k, const void* v, int S, int start_pos,
                           int Hq, int Hkv, int d, float scale, void* out,
                           cudaStream_t stream) {
  (void)d;
  const int T = start_pos + S;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, S, Hq) || !make_map(&mk, k, T, Hkv) || !make_map(&mv, v, T, Hkv))
    return cudaErrorInvalidValue;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tcgen05_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  PrefillParams p;
  p.out = static_cast<uint16_t*>(out);
  p.S = S;
  p.start_pos = start_pos;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.n_qt = (S + kBM - 1) / kBM;
  p.scale_log2 = scale * 1.4426950408889634f;
  const long long blocks = (long long)p.n_qt * Hq;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  prefill_tcgen05_kernel<<<(unsigned)blocks, kPThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace gqa
