// decode_tc.cuh -- split-KV decode attention with both contractions of a
// tile on the tcgen05 tensor cores, for g = 16 and for g = 8 with the rotary
// embedding (whose rotated query takes 16 operand rows); every other g <= 8
// runs on per-warp mma.sync MMAs (decode_kernels.cuh), which measured faster
// there.  The kernels and their launch, included by decode_g8.cu and
// decode_g16.cu.
//
// What it computes ("MiniCPM4 `forward_step` Attention Performance Fix",
// sections 3 and 4.1): for every sequence b and query head h,
//   out[b,h,:] = softmax_j(scale * q[b,h,:] . K[b,h/g,j,:]) V[b,h/g,j,:]
// over cache rows j = 0..positions[b] only (or the last W of them with a
// local window), optionally after appending the step's new K/V row (rotated
// by the rotary embedding if asked) and optionally advancing every position
// by one afterwards -- the same operation and options as the kernels of
// decode_kernels.cuh, whose segment walk, helpers and tensor maps this file
// shares.
//
// Why tensor cores: the g query heads of a KV head share every K and V row,
// so one 128-key tile is two small dense contractions,
//   S^T [128 keys x g] = K [128 x 128 dims] . Q^T [128 dims x g]
//   O^T [128 dims x g] += V^T [128 dims x 128 keys] . P^T [128 keys x g].
// On CUDA cores their multiply-adds, bf16 unpacking and lane reductions grow
// with g; at g = 8 they made a CUDA-core kernel issue-bound (0.66 of HBM on
// a large batch).  Here each is eight tcgen05.mma (M = 128, N = 16: the g
// heads padded to 16, K = 16), so a tile costs the CUDA cores only its
// softmax, and a large g = 8 batch streams at the copy rate.
//
// Layout per CTA (one per SM):
//  * warp 4, one thread: 2-D TMA loads (cp.async.bulk.tensor, 128-byte
//    swizzle) of each tile's K and V into a ring of 3 stages (2 where shared
//    memory is short), as two 64-dim column blocks each: exactly the
//    canonical K-major layout of K as the A operand of S^T, and the MN-major
//    layout of V as the A operand of O^T.
//  * warp 5, one thread: S^T_i into tensor memory (two buffers); warp 6,
//    one thread: O^T += V^T_i P^T_i once the softmax wrote P_i, which frees
//    the tile's stage.  Each blocks on its own barriers, so the softmax of
//    one tile overlaps the tensor core's work on the next.
//  * warps 0-3, thread t: key t of a tile (TMEM lane t of S^T) and dim t of
//    O^T.  A thread reads its key's g scores, the four warps agree on each
//    head's tile maximum through shared memory, and P (bf16) goes to shared
//    memory as the B operand of the next MMA.  The running maximum is raised
//    only when a head's maximum grows by more than 2^8 (O^T is then rescaled
//    in place); otherwise P may reach 2^8, harmless in bf16 and fp32.
//  * q is the B operand of S^T (bf16, exact).  With the rotary embedding the
//    rotated q (fp32) is split into bf16 high and low parts in rows g..2g-1,
//    and the two score columns are added, which keeps ~16 mantissa bits.
//  * The appended row (fused append) is left out of the tensor-core tile:
//    the CTA whose part ends the segment writes it to the cache and folds its
//    score and value (fp32, CUDA cores) into its partial at the end.  So no
//    load has to wait for that write.
//  * Segment splitting and merging follow decode_kernels.cuh (cluster mode:
//    partials pushed into rank 0's shared memory, here over contiguous tile
//    ranges; stream-K: partials through the workspace, merged by the last
//    CTA to arrive).
//  * Every wait is bounded (ATTN_DEV_TIMEOUT); the softmax warps' named
//    barriers sit where all four warps always arrive, whatever a wait gave.
#pragma once

#include "decode_kernels.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace {

constexpr int kTcN = 16;                       // MMA N: the g heads, padded
constexpr int kTcSW = 4;                       // softmax warps (TMEM lane quarters)
constexpr int kTcNC = kTcSW * 32;              // softmax threads
constexpr int kTcProdWarp = kTcSW;             // TMA
constexpr int kTcMmaWarp = kTcSW + 1;          // S^T MMAs, TMEM allocation
constexpr int kTcPvWarp = kTcSW + 2;           // O^T MMAs
constexpr int kTcThreads = (kTcSW + 3) * 32;
constexpr int kTcMaxStages = 3;                // K/V ring: 3 stages where shared memory allows, else 2
constexpr int kTcHalf = kTile * 128;           // 16 KB: 128 rows x 64 dims (one swizzle block)
constexpr int kTcOpBlock = kTcN * 128;         // 2 KB: 16 rows x 64 columns of Q or P
constexpr int kTcOpBytes = 2 * kTcOpBlock;     // a whole 16 x 128 operand
constexpr uint32_t kTcTmemCols = 64;
constexpr uint32_t kTcTmemS = 0;               // S^T of tile parity x: columns 16x .. 16x+15
constexpr uint32_t kTcTmemO = 32;              // O^T: columns 32 .. 47
constexpr float kTcTau = 8.0f;                 // a stale running max may lag by 2^8
// The rotation needs two operand rows per head (bf16 high and low parts of
// the rotated q): g <= 8.  g = 16 fills the 16 rows with plain q.
template <int G> constexpr bool kTcRope = 2 * G <= kTcN;

// mbarriers
constexpr int kTbFull = 0;                     // + stage: the tile's K and V landed
constexpr int kTbEmpty = kTbFull + kTcMaxStages;   // + stage: its MMAs are done with it
constexpr int kTbSFull = kTbEmpty + kTcMaxStages;  // + parity: S^T of a tile is in TMEM
constexpr int kTbPFull = kTbSFull + 2;         // + parity: P of a tile written (4 warps)
constexpr int kTbPVDone = kTbPFull + 2;        // + parity: O^T += V^T P^T of a tile done
constexpr int kTbQFull = kTbPVDone + 2;        // + parity: a segment's Q operand (4 warps)
constexpr int kTbOFree = kTbQFull + 2;         // the epilogue has read O^T (4 warps)
constexpr int kTbCount = kTbOFree + 1;

// Shared memory, from a 1024-byte aligned base: the ns K/V stages (64 KB
// each), then at fix = ns * 64 KB the parts below, then the tail (stream-K:
// the tile prefix sum [B+1]; cluster mode: rank 0's landing slots).
constexpr int kToQ = 0;                           // Q operand, two buffers (by segment)
constexpr int kToP = kToQ + 2 * kTcOpBytes;       // P operand, two buffers (by tile)
constexpr int kToBar = kToP + 2 * kTcOpBytes;
constexpr int kToMisc = kToBar + 128;
constexpr int kToRed = kToMisc + kMiscInts * 4;   // floats: tile maxima [2][4][16], sums [4][32]
constexpr int kToTail = kToRed + (2 * kTcSW * kTcN + kTcSW * 2 * kTcN) * 4;
static_assert(kTbCount * 8 <= 128, "mbarriers");
constexpr int kTcMaxSmem = 232448;                // per-block opt-in maximum (227 KB)
// misc ints: [0] abort, [1] last-arrival flag, [4] TMEM address, [8..12) scan

// Byte offset of element (r, c) of a 16-row operand (Q or P: row = head,
// column = dim or key), K-major in the 128-byte swizzled layout: column block
// c/64, 128-byte row r, 16-byte chunk (c%64)/8 XOR r%8.
__device__ __forceinline__ uint32_t op_off(int r, int c) {
  return (uint32_t)((c >> 6) * kTcOpBlock + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                    (c & 7) * 2);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const __nv_bfloat16 r = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&r);
}
__device__ __forceinline__ float bf16_val(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

// Reduction (max or sum) over the 32 lanes of G values at once.  A step with
// offset `off` keeps half of the values and ships the other half to the
// partner lane, so after log2(G) steps each lane carries one value index,
// lane >> (5 - log2 G); the remaining steps are a plain butterfly.
template <int G, bool MAX>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[G], int lane) {
  constexpr int LG = Log2<G>::v;
#pragma unroll
  for (int st = 0; st < LG; ++st) {
    const int off = 16 >> st;
    const int n = G >> (st + 1);
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = upper ? v[n + i] : v[i];
      const float send = upper ? v[i] : v[n + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float x = v[0];
#pragma unroll
  for (int off = 16 >> LG; off >= 1; off >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, x, off);
    x = MAX ? fmaxf(x, got) : x + got;
  }
  return x;
}

// The four softmax warps only.  Every softmax warp reaches each of these
// barriers on every path (their loops have the same trip counts and no
// early exit), so none can wait for ever.
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Non-blocking test of an mbarrier phase (try_wait may suspend the thread for
// a while, which would hold up a thread polling several barriers).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// One thread's bounded wait; on failure it raises the abort flag.
__device__ __forceinline__ bool lane_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
  if (mbar_wait(bar, parity, abort_flag)) return true;
  *abort_flag = 1;
  set_status(status, ATTN_DEV_TIMEOUT);
  return false;
}

// Thread d of the softmax warps writes dim d of the segment's Q operand: the
// G query rows (rotated, as bf16 high and low parts, with the rotary
// embedding at position pos).
template <int G, int M>
__device__ __forceinline__ void write_q_operand(const Params& p, uint8_t* q_op, int b, int kvh,
                                                int pos, int d) {
  constexpr bool R = (M & kModeRope) != 0, MT = (M & kModeMulti) != 0;
  const float* rc = rope_row<R>(p, p.rope_cos, b, pos);
  const float* rs = rope_row<R>(p, p.rope_sin, b, pos);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint16_t* qh = p.q + head_row<G, MT>(p, b, kvh, h) * kD;
    const uint16_t x = qh[d];
    if (R) {
      const float xr = rope1(bf16_val(x), bf16_val(qh[d ^ (kD / 2)]), rc[d], rs[d], d < kD / 2);
      const uint16_t hi = bf16_bits(xr);
      *reinterpret_cast<uint16_t*>(q_op + op_off(h, d)) = hi;
      *reinterpret_cast<uint16_t*>(q_op + op_off(G + h, d)) = bf16_bits(xr - bf16_val(hi));
    } else {
      *reinterpret_cast<uint16_t*>(q_op + op_off(h, d)) = x;
    }
  }
}

template <bool CL>
__device__ __forceinline__ void tiles_next(Walk& w, const Params& p, const int* prefix, int win,
                                           int shift) {
  if (CL) ++w.k;
  else walk_next(w, prefix, p.positions, p.B, p.Hkv, win, shift);
}

// Dynamic shared memory of a launch with ns stages: stream-K (C = 0) for a
// batch of B, or cluster mode with clusters of C.
template <int G>
size_t tc_smem_bytes(int ns, int C, int B) {
  return 1024 + (size_t)ns * 2 * kTileBytes + kToTail +
         (C > 0 ? (size_t)C * G * (kD + 2) * sizeof(float) : (size_t)(B + 1) * sizeof(int));
}

// CL: cluster mode (grid = B*Hkv clusters of C CTAs, cluster s = segment s);
// otherwise stream-K over a persistent grid.
template <int G, int M, bool CL>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params p, const int ns) {
  constexpr bool R = (M & kModeRope) != 0, A = (M & kModeAdvance) != 0;
  constexpr bool MT = (M & kModeMulti) != 0;
  static_assert((R ? 2 * G : G) <= kTcN, "Q operand rows");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int fix = ns * 2 * kTileBytes;  // after the stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + fix + kToBar);
  int* misc = reinterpret_cast<int*>(smem + fix + kToMisc);
  float* tmax = reinterpret_cast<float*>(smem + fix + kToRed);  // [2][kTcSW][kTcN]
  float* red = tmax + 2 * kTcSW * kTcN;                    // [kTcSW][2 * kTcN]
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, L = p.L;
  const int win = (M & kModeWindow) ? p.window : 0;
  const int shift = MT ? p.S - 1 : 0;  // positions[b] + shift: the last new token's row
  volatile int* abort_flag = misc;

  // The TMA thread initialises the mbarriers itself, so it may start loading
  // as soon as it knows its tiles; everyone else sees them after the setup
  // barrier below.
  const bool tma_thread = warp == kTcProdWarp && lane == 0;
  if (tma_thread) {
#pragma unroll
    for (int s = 0; s < kTcMaxStages; ++s) {
      mbar_init(bar(kTbFull + s), 1);   // the TMA thread's arrival + bytes
      mbar_init(bar(kTbEmpty + s), 1);  // tcgen05.commit
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kTbSFull + x), 1);
      mbar_init(bar(kTbPFull + x), kTcSW);
      mbar_init(bar(kTbPVDone + x), 1);
      mbar_init(bar(kTbQFull + x), kTcSW);
    }
    mbar_init(bar(kTbOFree), kTcSW);
    misc[0] = 0;
    misc[1] = 0;
    fence_mbar_init();
  }
  // Launched with programmatic stream serialisation: nothing the previous
  // kernel on the stream wrote is read before this wait.
  grid_dependency_wait();
  grid_dependents_launch();

  // ---- this CTA's tiles: `count` tiles from w0 ------------------------------
  Walk w0;
  int count = 0;
  int* prefix = reinterpret_cast<int*>(smem + fix + kToTail);  // stream-K: [B+1]
  long long t0 = 0, T = 0;
  int Gd = 1, C = 1, rank = 0;
  if constexpr (CL) {
    cg::cluster_group cluster = cg::this_cluster();
    C = (int)cluster.num_blocks();
    rank = (int)cluster.block_rank();
    const int seg = blockIdx.x / C;
    const int b = seg / Hkv, kvh = seg % Hkv;
    const int pos0 = p.positions[b];
    if (!rows_in_cache(pos0, shift, L)) {
      // the same for every CTA of the cluster: all leave, no cluster barrier
      if (rank == 0 && kvh == 0 && tid == 0) {
        set_status(p.status, ATTN_DEV_BAD_POSITION);
        write_nan_rows(p, b, MT ? p.S : 1);
      }
      if (A) {
        __syncthreads();  // every thread's read of positions is done
        if (warp == 0) advance_ticket(p, lane);
      }
      return;
    }
    int lo, n;
    attended_rows(pos0 + shift, win, lo, n);
    const int ntiles = (n - 1) / kTile + 1;
    const int k0 = (int)((long long)rank * ntiles / C);
    const int k1 = (int)((long long)(rank + 1) * ntiles / C);
    w0.b = b;
    w0.kvh = kvh;
    w0.k = k0;
    w0.ntiles = ntiles;
    w0.n = n;
    w0.lo = lo;
    count = k1 - k0;
  } else {
    // tiles per sequence and their exclusive prefix sum (every CTA)
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += kTcNC) {
      const int b = b0 + tid;
      int v = 0;
      if (tid < kTcNC && b < B) {
        const int p0 = p.positions[b];
        if (rows_in_cache(p0, shift, L)) {
          int lo, n;
          attended_rows(p0 + shift, win, lo, n);
          v = (n - 1) / kTile + 1;
        } else if (b % gridDim.x == blockIdx.x) {
          set_status(p.status, ATTN_DEV_BAD_POSITION);
          write_nan_rows(p, b, MT ? p.S : 1);
        }
      }
      int x = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (lane == 31 && warp < kTcSW) misc[8 + warp] = x;
      __syncthreads();
      int before = 0, chunk = 0;
#pragma unroll
      for (int ww = 0; ww < kTcSW; ++ww) {
        const int s = misc[8 + ww];
        before += (ww < warp) ? s : 0;
        chunk += s;
      }
      if (tid < kTcNC && b < B) prefix[b] = carry + before + x - v;
      carry += chunk;
      __syncthreads();
    }
    if (tid == 0) prefix[B] = carry;
    __syncthreads();
    T = (long long)Hkv * carry;
    // one CTA per segment when segments are short (a split costs a partial
    // round trip through L2); never more CTAs than tiles
    const long long nseg = (long long)B * Hkv;
    long long gw = min((long long)gridDim.x, T);
    if (T <= (long long)kWholeTiles * nseg) gw = min(gw, nseg);
    Gd = (int)gw;
    if ((int)blockIdx.x >= Gd) {  // every thread is past its reads of positions
      if (A && warp == 0) advance_ticket(p, lane);
      return;
    }
    t0 = T * blockIdx.x / Gd;
    const long long t1 = T * (blockIdx.x + 1) / Gd;
    count = (int)(t1 - t0);
    walk_init(w0, t0, prefix, p.positions, B, Hkv, win, shift);
  }

  // ---- the first loads, before the rest of the setup -------------------------
  Walk pw = w0;         // TMA thread: next tile to load,
  int pi = 0, ps = 0;   //   its index and stage,
  uint32_t pu = 0;      //   and index / ns
  auto produce_until = [&](int i_end) {
    for (; pi < i_end; ++pi) {
      if (pi >= ns && !lane_wait(bar(kTbEmpty + ps), (pu & 1u) ^ 1u, abort_flag, p.status)) {
        pi = count;
        break;
      }
      // failure-path tests only: tile test_skip of the first segment is
      // never issued, so the bounded waits for it run out
      if (!(p.test_skip >= 0 && pw.b == 0 && pw.kvh == 0 && pw.k == p.test_skip)) {
        const uint32_t full = bar(kTbFull + ps);
        const uint32_t sK = base + (uint32_t)(ps * 2 * kTileBytes);
        const int row = pw.lo + pw.k * kTile, z = pw.b * Hkv + pw.kvh;
        if (range_ok(z >= 0 && z < p.B * Hkv && row >= 0 && row < L, p.status)) {
          mbar_arrive_expect_tx(full, 2u * kTileBytes);
          tma_load_3d(sK, &tm_k, 0, row, z, full);
          tma_load_3d(sK + kTcHalf, &tm_k, 64, row, z, full);
          tma_load_3d(sK + kTileBytes, &tm_v, 0, row, z, full);
          tma_load_3d(sK + kTileBytes + kTcHalf, &tm_v, 64, row, z, full);
        }
      }
      tiles_next<CL>(pw, p, prefix, win, shift);
      if (++ps == ns) {
        ps = 0;
        ++pu;
      }
    }
  };
  if (tma_thread) produce_until(min(ns, count));  // no stage to wait for yet

  // ---- tensor memory, operand buffers -------------------------------------
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc + 4);
  if (warp == kTcMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kTcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // rows of Q and P no writer touches hold zeros (finite) for good
  for (int i = tid; i < 4 * kTcOpBytes / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(smem + fix + kToQ)[i] = make_uint4(0u, 0u, 0u, 0u);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if constexpr (CL) {
    // this CTA runs: the matching wait comes before any write into rank 0's
    // shared memory, so rank 0 is known to have started by then
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  }
  float* land_o = reinterpret_cast<float*>(smem + fix + kToTail);  // cluster: [C][G][kD]
  float* land_ml = land_o + C * G * kD;                              //          [C][G][2]

  if (warp == kTcProdWarp) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) produce_until(count);
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------- S^T = K Q^T --
    // One thread per MMA stream, each blocking on its own barriers (a thread
    // polling several would steal issue slots from the softmax warp that
    // shares its scheduler).  Tile nq needs its K/V landed, its segment's Q
    // written, and S buffer nq&1 free: the softmax is past tile nq-2.
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, kTcN, false);
      Walk w = w0;
      int j = -1, s = 0;
      uint32_t u = 0;
      for (int nq = 0; nq < count; ++nq) {
        const bool first = (nq == 0) || w.k == 0;
        if (first) ++j;
        if (first &&
            !lane_wait(bar(kTbQFull + (j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, p.status))
          break;
        if (!lane_wait(bar(kTbFull + s), u & 1u, abort_flag, p.status)) break;
        if (nq >= 2 && !lane_wait(bar(kTbPFull + (nq & 1)), (uint32_t)((nq - 2) >> 1) & 1u,
                                  abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t sK = base + (uint32_t)(s * 2 * kTileBytes);
        const uint32_t sQ = base + (uint32_t)(fix + kToQ + (j & 1) * kTcOpBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)  // 4 K-steps per 64-dim column block
          tc_mma(tmem + kTcTmemS + (uint32_t)((nq & 1) * kTcN),
                 sw128_desc(sK + (kk >> 2) * kTcHalf + (kk & 3) * 32),
                 sw128_desc(sQ + (kk >> 2) * kTcOpBlock + (kk & 3) * 32), idesc_s,
                 kk > 0 ? 1u : 0u);
        tc_commit(bar(kTbSFull + (nq & 1)));
        tiles_next<CL>(w, p, prefix, win, shift);
        if (++s == ns) {
          s = 0;
          ++u;
        }
      }
    }
    __syncwarp();
  } else if (warp == kTcPvWarp) {
    // ---------------------------------------------------- O^T += V^T P^T --
    // Tile np needs its P written (so its S^T, and the K half of its stage,
    // are done with) and, first in a segment, the previous segment's
    // epilogue done reading O^T.  Its completion frees the stage.
    if (lane == 0) {
      constexpr uint32_t idesc_o = make_idesc(128, kTcN, false, true);  // V^T: MN-major
      Walk w = w0;
      int j = -1, s = 0;
      for (int np = 0; np < count; ++np) {
        const bool first = (np == 0) || w.k == 0;
        if (first) ++j;
        if (!lane_wait(bar(kTbPFull + (np & 1)), (uint32_t)(np >> 1) & 1u, abort_flag, p.status))
          break;
        if (first && j > 0 &&
            !lane_wait(bar(kTbOFree), (uint32_t)(j - 1) & 1u, abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t sV = base + (uint32_t)(s * 2 * kTileBytes + kTileBytes);
        const uint32_t sP = base + (uint32_t)(fix + kToP + (np & 1) * kTcOpBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma(tmem + kTcTmemO, sw128_desc(sV + kk * 16 * 128, kTcHalf),
                 sw128_desc(sP + (kk >> 2) * kTcOpBlock + (kk & 3) * 32), idesc_o,
                 (first && kk == 0) ? 0u : 1u);
        tc_commit(bar(kTbPVDone + (np & 1)));
        tc_commit(bar(kTbEmpty + s));  // the stage may be refilled
        tiles_next<CL>(w, p, prefix, win, shift);
        if (++s == ns) s = 0;
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- softmax --
    const int t = tid;  // key t of a tile; dim t of O^T
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + kTcTmemS + lane_off;
    const uint32_t tO = tmem + kTcTmemO + lane_off;
    const float qs = p.qscale;
    constexpr int LG = Log2<G>::v;
    float m_ref[G], l_t[G];
    int head_last[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_ref[h] = -INFINITY;
      l_t[h] = 0.f;
      head_last[h] = 0;
    }
    // the appended row, loaded at its segment's start and used at the end:
    // k and v at dim t (k's partner dim for the rotation), q of each head
    uint16_t fk = 0, fk2 = 0, fv = 0, fq[G], fq2[G];
    float frc = 0.f, frs = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) fq[h] = fq2[h] = 0;
    bool ok = true;
    Walk w = w0;
    int j = 0;
    if (count > 0) {
      write_q_operand<G, M>(p, smem + fix + kToQ, w.b, w.kvh, w.lo + w.n - 1, t);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kTbQFull));
    }
    for (int i = 0; i < count; ++i) {
      const bool first = (i == 0) || w.k == 0;
      if (i > 0 && first) ++j;
      const bool last_of_seg = w.k == w.ntiles - 1;
      const bool seg_end = last_of_seg || i == count - 1;
      if (MT && first) {
#pragma unroll
        for (int h = 0; h < G; ++h) head_last[h] = w.lo + w.n - 1 - shift + h / (G / p.S);
      }
      float sv[kTcN];
      ok = ok && consumer_wait(bar(kTbSFull + (i & 1)), (uint32_t)(i >> 1) & 1u, abort_flag,
                               p.status, lane);
      if (ok) {
        tc_fence_after();
        tmem_ld16(tS + (uint32_t)((i & 1) * kTcN), sv);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int c = 0; c < kTcN; ++c) sv[c] = 0.f;
      }
      if (!CL && first) {
        // the next segment's Q into the other buffer: this S^T wait means
        // every MMA of the segment before, which read that buffer, is done
        const long long tn = t0 + i + (w.ntiles - w.k);
        if (tn < t0 + count) {
          Walk nw;
          walk_init(nw, tn, prefix, p.positions, B, Hkv, win, shift);
          write_q_operand<G, M>(p, smem + fix + kToQ + ((j + 1) & 1) * kTcOpBytes, nw.b, nw.kvh,
                                nw.lo + nw.n - 1, t);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kTbQFull + ((j + 1) & 1)));
        }
      }
      if (first && p.k_new != nullptr && i + (w.ntiles - 1 - w.k) < count) {
        // this CTA's part ends the segment, so the appended row is its own:
        // start its loads now, use them in the epilogue
        const size_t src = ((size_t)w.b * Hkv + w.kvh) * kD;
        const uint16_t* kn = reinterpret_cast<const uint16_t*>(p.k_new) + src;
        fk = kn[t];
        fv = reinterpret_cast<const uint16_t*>(p.v_new)[src + t];
#pragma unroll
        for (int h = 0; h < G; ++h) fq[h] = p.q[head_row<G, MT>(p, w.b, w.kvh, h) * kD + t];
        if (R) {
          const int pos = w.lo + w.n - 1;
          fk2 = kn[t ^ (kD / 2)];
#pragma unroll
          for (int h = 0; h < G; ++h)
            fq2[h] = p.q[head_row<G, MT>(p, w.b, w.kvh, h) * kD + (t ^ (kD / 2))];
          frc = rope_row<R>(p, p.rope_cos, w.b, pos)[t];
          frs = rope_row<R>(p, p.rope_sin, w.b, pos)[t];
        }
      }
      const int rows = min(kTile, w.n - w.k * kTile);
      const bool fresh = p.k_new != nullptr && last_of_seg;  // appended row: folded in later
      const int rows_mma = rows - (fresh ? 1 : 0);
      const int row0 = w.lo + w.k * kTile;
      float s[G], mx[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float x = (R ? sv[h] + sv[G + h] : sv[h]) * qs;
        const bool valid = t < rows_mma && (!MT || row0 + t <= head_last[h]);
        s[h] = valid ? x : -INFINITY;
        mx[h] = s[h];
      }
      const float hm = warp_reduce_heads<G, true>(mx, lane);
      if ((lane & ((32 >> LG) - 1)) == 0)
        tmax[((i & 1) * kTcSW + warp) * kTcN + (lane >> (5 - LG))] = hm;
      softmax_bar();
      bool grow_any = false;
      float Mt[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a = tmax[((i & 1) * kTcSW) * kTcN + h];
#pragma unroll
        for (int ww = 1; ww < kTcSW; ++ww) a = fmaxf(a, tmax[((i & 1) * kTcSW + ww) * kTcN + h]);
        Mt[h] = a;
        grow_any = grow_any || a > m_ref[h] + kTcTau;
      }
      if (grow_any) {  // the same decision in every softmax thread
        float alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const bool gr = Mt[h] > m_ref[h] + kTcTau;
          alpha[h] = gr ? ex2(m_ref[h] - Mt[h]) : 1.f;  // m_ref = -inf: 0
          m_ref[h] = gr ? Mt[h] : m_ref[h];
          l_t[h] *= alpha[h];
        }
        if (!first) {  // O^T holds this segment's tiles so far: rescale it
          ok = ok && consumer_wait(bar(kTbPVDone + ((i - 1) & 1)), (uint32_t)((i - 1) >> 1) & 1u,
                                   abort_flag, p.status, lane);
          if (ok) {
            tc_fence_after();
            float o[kTcN];
            tmem_ld16(tO, o);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] *= alpha[h];
            tmem_st16(tO, o);
            tmem_st_wait();
          }
        }
      }
      // P buffer i&1 is free once the O^T update of tile i-2 is done
      if (i >= 2)
        ok = ok && consumer_wait(bar(kTbPVDone + (i & 1)), (uint32_t)((i - 2) >> 1) & 1u,
                                 abort_flag, p.status, lane);
      if (ok) {
        uint8_t* Pb = smem + fix + kToP + (i & 1) * kTcOpBytes;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float m_use = (m_ref[h] == -INFINITY) ? 0.f : m_ref[h];  // no valid key yet
          const uint16_t pb = bf16_bits(ex2(s[h] - m_use));
          *reinterpret_cast<uint16_t*>(Pb + op_off(h, t)) = pb;
          l_t[h] += bf16_val(pb);
        }
        if (last_of_seg && rows_mma < kTile) {
          // rows past the segment (or the appended row) hold whatever the
          // cache has there: zero V's row, since its P of 0 times NaN would
          // not be 0.  After the tile's own landing, which this wait shows.
          ok = consumer_wait(bar(kTbFull + i % ns), (uint32_t)(i / ns) & 1u, abort_flag,
                             p.status, lane);
          uint4* vr = reinterpret_cast<uint4*>(smem + (i % ns) * 2 * kTileBytes + kTileBytes +
                                               t * 128);
          if (ok && t >= rows_mma) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int cc = (c + t) & 7;  // spread the lanes over the banks
              vr[cc] = make_uint4(0u, 0u, 0u, 0u);
              vr[kTcHalf / 16 + cc] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kTbPFull + (i & 1)));

      if (seg_end) {
        // ---- this CTA's part of the segment: O^T -> partial or output -----
        float o[kTcN];
        ok = ok && consumer_wait(bar(kTbPVDone + (i & 1)), (uint32_t)(i >> 1) & 1u, abort_flag,
                                 p.status, lane);
        if (ok) {
          tc_fence_after();
          tmem_ld16(tO, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < kTcN; ++c) o[c] = 0.f;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kTbOFree));

        // the appended row: written to the cache, then its score and value
        // join this partial
        // the appended row: to the cache (no load of this launch read it:
        // the tile holding it masked that row), and q.k per head
        float vals[2 * G];
        float vd = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          vals[h] = l_t[h];
          vals[G + h] = 0.f;
        }
        if (fresh) {
          const int pos = w.lo + w.n - 1;
          const uint16_t kb =
              R ? bf16_bits(rope1(bf16_val(fk), bf16_val(fk2), frc, frs, t < kD / 2)) : fk;
          const size_t dst = (((size_t)w.b * Hkv + w.kvh) * (size_t)L + (size_t)pos) * kD + t;
          reinterpret_cast<uint16_t*>(p.k_cache)[dst] = kb;
          reinterpret_cast<uint16_t*>(p.v_cache)[dst] = fv;
          const float kf = bf16_val(kb);
          vd = bf16_val(fv);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float qv = R ? rope1(bf16_val(fq[h]), bf16_val(fq2[h]), frc, frs, t < kD / 2)
                               : bf16_val(fq[h]);
            vals[G + h] = qv * kf;
          }
        }
        {
          constexpr int LV = Log2<2 * G>::v;
          const float hs = warp_reduce_heads<2 * G, false>(vals, lane);
          if ((lane & ((32 >> LV) - 1)) == 0) red[warp * 2 * kTcN + (lane >> (5 - LV))] = hs;
        }
        softmax_bar();
        float mo[G], lo_[G], oo[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float Ls = 0.f, dot = 0.f;
#pragma unroll
          for (int ww = 0; ww < kTcSW; ++ww) {
            Ls += red[ww * 2 * kTcN + h];
            dot += red[ww * 2 * kTcN + G + h];
          }
          float m = m_ref[h], oh = o[h];
          if (fresh) {
            const float sf = dot * qs;
            const float Mx = fmaxf(m, sf);
            const float a = ex2(m - Mx), e = ex2(sf - Mx);  // m = -inf: a = 0
            oh = oh * a + e * vd;
            Ls = Ls * a + e;
            m = Mx;
          }
          mo[h] = m;
          lo_[h] = Ls;
          oo[h] = oh;
        }

        if constexpr (CL) {
          asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
          cg::cluster_group cluster = cg::this_cluster();
          float* to_o = cluster.map_shared_rank(land_o, 0) + rank * G * kD;
          float* to_ml = cluster.map_shared_rank(land_ml, 0) + rank * G * 2;
          const bool land_ok = range_ok(rank < kMaxCluster && C <= kMaxCluster, p.status);
#pragma unroll
          for (int h = 0; h < G && land_ok; ++h) {
            to_o[h * kD + t] = oo[h];
            if (t == 0) {
              to_ml[h * 2 + 0] = mo[h];
              to_ml[h * 2 + 1] = lo_[h];
            }
          }
        } else {
          const int seg = w.b * Hkv + w.kvh;
          const long long seg_t0 = (long long)Hkv * prefix[w.b] + (long long)w.kvh * w.ntiles;
          const long long seg_t1 = seg_t0 + w.ntiles;
          const bool whole = seg_t0 >= t0 && seg_t1 <= t0 + count;
          if (whole) {
#pragma unroll
            for (int h = 0; h < G; ++h)
              store_out(p, head_row<G, MT>(p, w.b, w.kvh, h), t, oo[h] / lo_[h]);
          } else {
            const int slot = blockIdx.x + seg;
            const bool slot_ok = range_ok(slot < kMaxGrid + B * Hkv, p.status);
#pragma unroll
            for (int h = 0; h < G && slot_ok; ++h) {
              p.part_o[((size_t)slot * G + h) * kD + t] = oo[h];
              if (t == 0) {
                p.part_ml[((size_t)slot * G + h) * 2 + 0] = mo[h];
                p.part_ml[((size_t)slot * G + h) * 2 + 1] = lo_[h];
              }
            }
            const int c_first = cta_of(seg_t0, T, Gd);
            const int c_last = cta_of(seg_t1 - 1, T, Gd);
            softmax_bar();  // every partial store of this CTA comes before the ticket
            if (t == 0) {
              // release: this CTA's partial is visible to whoever acquires
              // the counter; acquire: the last arrival sees every other's
              unsigned old;
              asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                           : "=r"(old)
                           : "l"(&p.counters[seg])
                           : "memory");
              misc[1] = (old == (unsigned)(c_last - c_first)) ? 1 : 0;
            }
            softmax_bar();
            if (misc[1]) {
              // last to arrive: merge the segment's partials, batches of 8
              // independent loads in flight
              for (int idx = t; idx < G * kD; idx += kTcNC) {
                const int h = idx / kD, d = idx % kD;
                float Mm = -INFINITY, Ls = 0.f, Os = 0.f;
                for (int c0 = c_first; c0 <= c_last; c0 += 8) {
                  float mm[8], ll[8], ov[8];
#pragma unroll
                  for (int uu = 0; uu < 8; ++uu) {
                    const int c = c0 + uu;
                    if (c <= c_last && range_ok(c + seg < kMaxGrid + B * Hkv, p.status)) {
                      const size_t sl = (size_t)(c + seg) * G + h;
                      mm[uu] = __ldcg(&p.part_ml[sl * 2]);
                      ll[uu] = __ldcg(&p.part_ml[sl * 2 + 1]);
                      ov[uu] = __ldcg(&p.part_o[sl * kD + d]);
                    } else {
                      mm[uu] = -INFINITY;
                      ll[uu] = 0.f;
                      ov[uu] = 0.f;
                    }
                  }
                  float Mb = Mm;
#pragma unroll
                  for (int uu = 0; uu < 8; ++uu) Mb = fmaxf(Mb, mm[uu]);
                  const float sc0 = ex2(Mm - Mb);  // Mm = -inf on the first batch: 0
                  Ls *= sc0;
                  Os *= sc0;
#pragma unroll
                  for (int uu = 0; uu < 8; ++uu) {
                    const float e = ex2(mm[uu] - Mb);
                    Ls = fmaf(ll[uu], e, Ls);
                    Os = fmaf(ov[uu], e, Os);
                  }
                  Mm = Mb;
                }
                store_out(p, head_row<G, MT>(p, w.b, w.kvh, h), d, Os / Ls);
              }
              if (t == 0) p.counters[seg] = 0u;  // ready for the next launch
            }
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m_ref[h] = -INFINITY;
          l_t[h] = 0.f;
        }
      }
      tiles_next<CL>(w, p, prefix, win, shift);
    }
    if constexpr (CL) {
      if (count == 0) {
      // no tiles: an empty partial (max -inf, sum 0, o 0)
      asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
      cg::cluster_group cluster = cg::this_cluster();
      float* to_o = cluster.map_shared_rank(land_o, 0) + rank * G * kD;
      float* to_ml = cluster.map_shared_rank(land_ml, 0) + rank * G * 2;
      const bool land_ok = range_ok(rank < kMaxCluster && C <= kMaxCluster, p.status);
#pragma unroll
      for (int h = 0; h < G && land_ok; ++h) {
        to_o[h * kD + t] = 0.f;
        if (t == 0) {
          to_ml[h * 2 + 0] = -INFINITY;
          to_ml[h * 2 + 1] = 0.f;
        }
      }
      }
    }
  }

  if constexpr (CL) {
    if (warp >= kTcSW) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every rank's partial is in rank 0's shared memory
    if (rank == 0) {
      // weights 2^(m_r - M) / L per (rank, head): a warp per head reduces
      // over the ranks, lane r holding rank r's (max, sum)
      static_assert(kMaxCluster * G <= 2 * kTcSW * kTcN + kTcSW * 2 * kTcN,
                    "the weights fit the tile-maxima and sums buffers");
      float* wr = tmax;  // [C][G], over tmax and red (both free by now)
      for (int h = warp; h < G; h += kTcThreads / 32) {
        const bool in = lane < C;
        const float m = in ? land_ml[(lane * G + h) * 2] : -INFINITY;
        const float l = in ? land_ml[(lane * G + h) * 2 + 1] : 0.f;
        float Mx = m;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
        const float e = in ? ex2(m - Mx) : 0.f;  // a rank without keys: 2^-inf = 0
        float Ls = l * e;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
        if (in) wr[lane * G + h] = e / Ls;
      }
      __syncthreads();
      for (int idx = tid; idx < G * kD; idx += kTcThreads) {
        const int h = idx / kD, d = idx % kD;
        float Os = 0.f;
#pragma unroll 4
        for (int r = 0; r < C; ++r) Os = fmaf(land_o[(r * G + h) * kD + d], wr[r * G + h], Os);
        store_out(p, head_row<G, MT>(p, w0.b, w0.kvh, h), d, Os);
      }
    }
    // no second cluster barrier: no CTA reads another's shared memory again
  }

  // ------------------------------------------------------------ teardown --
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let copies and tensor-core work still in flight land before TMEM goes
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
  }
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTcTmemCols)
                 : "memory");
  }
  // every thread read positions only before the barrier above
  if (A && warp == 0) advance_ticket(p, lane);
}

// ------------------------------------------------------------------ host --

struct TcDevInfo {
  bool configured[17] = {};                // per g (8 and 16)
  int clusters[17][kMaxCluster + 1] = {};  // [g][C]: co-resident clusters of C CTAs
};
TcDevInfo g_tc_dev[64];

template <int G>
int tc_max_clusters(int C) {
  // rank 0 holds a landing slot per rank: at g = 16 that limits C to 9
  if (tc_smem_bytes<G>(2, C, 0) > (size_t)kTcMaxSmem) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C * 64);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = tc_smem_bytes<G>(2, C, 0);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<G, 0, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int G, int M>
cudaError_t tc_set_attributes(bool* big) {
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G, M, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_tc_kernel<G, M, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem);
  if (e != cudaSuccess) return e;
  *big = cudaFuncSetAttribute(decode_tc_kernel<G, M, true>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (!*big) cudaGetLastError();
  return cudaSuccess;
}

template <int G>
cudaError_t tc_configure(TcDevInfo& d) {
  if (d.configured[G]) return cudaSuccess;
  bool big[6] = {true, true, true, true, true, true};
  cudaError_t e = tc_set_attributes<G, 0>(&big[0]);
  if constexpr (kTcRope<G>) {
    if (e == cudaSuccess) e = tc_set_attributes<G, kModeRope>(&big[1]);
    if (e == cudaSuccess) e = tc_set_attributes<G, kModeRope | kModeAdvance>(&big[3]);
  }
  if (e == cudaSuccess) e = tc_set_attributes<G, kModeAdvance>(&big[2]);
  if (e == cudaSuccess) e = tc_set_attributes<G, kModeWindow>(&big[4]);
  if (e == cudaSuccess) e = tc_set_attributes<G, kModeMulti>(&big[5]);
  if (e != cudaSuccess) return e;
  const bool big_all = big[0] && big[1] && big[2] && big[3] && big[4] && big[5];
  // A cluster stays within one GPC, so how many fit at once is set by the SMs
  // per GPC, not by the SM count.  All variants share block, shared memory and
  // registers, so the plain one stands for all.
  for (int c = 2; c <= kMaxCluster; ++c)
    d.clusters[G][c] = (c <= 8 || big_all) ? tc_max_clusters<G>(c) : 0;
  d.configured[G] = true;
  return cudaSuccess;
}

template <int G, int M>
cudaError_t launch_tc_g(const Params& p, cudaStream_t stream) {
  int dev = 0;
  DevInfo& di = dev_info(&dev);
  TcDevInfo& d = g_tc_dev[dev];
  cudaError_t e = tc_configure<G>(d);
  if (e != cudaSuccess) return e;
  const long long nseg = (long long)p.B * p.Hkv;
  CUtensorMap mk, mv;
  if (!cache_map(&mk, p.k_cache, p.L, nseg) || !cache_map(&mv, p.v_cache, p.L, nseg))
    return cudaErrorInvalidValue;
  // Cluster mode when every segment can have its own co-resident cluster of
  // at least 8 CTAs: the largest such size.  Otherwise stream-K.
  int C = 0;
  for (int c = kMaxCluster; c >= 8 && C == 0; --c)
    if (nseg <= d.clusters[G][c]) C = c;
  const int force = g_decode_test_cluster;  // schedule tests only
  if (force >= 0) {
    // a cluster size this kernel cannot launch is refused, not replaced
    if (force > kMaxCluster || tc_smem_bytes<G>(2, force, 0) > (size_t)kTcMaxSmem ||
        (force > 8 && d.clusters[G][force] == 0))
      return cudaErrorNotSupported;
    C = force;
  }
  // three K/V stages when they fit in shared memory, else two
  auto stages = [&](int c, int b) { return tc_smem_bytes<G>(3, c, b) <= (size_t)kTcMaxSmem ? 3 : 2; };
  if (C > 0) {
    const int ns = stages(C, 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nseg * C));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = tc_smem_bytes<G>(ns, C, 0);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<G, M, true>, mk, mv, p, ns);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const int ns = stages(0, p.B);
  return launch_pdl(decode_tc_kernel<G, M, false>, dim3(min(kMaxGrid, di.num_sms)),
                    dim3(kTcThreads), tc_smem_bytes<G>(ns, 0, p.B), stream, mk, mv, p, ns);
}

// The variant for this launch (the same six combinations as the kernels of
// decode_kernels.cuh).
template <int G>
cudaError_t launch_group_tc(const Params& p, cudaStream_t stream) {
  const int mode = (p.rope_cos != nullptr ? kModeRope : 0) |
                   (p.advance != nullptr ? kModeAdvance : 0) | (p.window > 0 ? kModeWindow : 0) |
                   (p.S > 1 ? kModeMulti : 0);
  if constexpr (kTcRope<G>) {
    if (mode == kModeRope) return launch_tc_g<G, kModeRope>(p, stream);
    if (mode == (kModeRope | kModeAdvance))
      return launch_tc_g<G, kModeRope | kModeAdvance>(p, stream);
  }
  switch (mode) {
    case 0: return launch_tc_g<G, 0>(p, stream);
    case kModeAdvance: return launch_tc_g<G, kModeAdvance>(p, stream);
    case kModeWindow: return launch_tc_g<G, kModeWindow>(p, stream);
    case kModeMulti: return launch_tc_g<G, kModeMulti>(p, stream);
  }
  return cudaErrorInvalidValue;  // a combination no entry point makes, or the
                                 // rotation at g = 16 (the entry points refuse it)
}

}  // namespace
}  // namespace gqa
