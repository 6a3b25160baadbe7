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
// How: work items are (pair of 128-token query tiles, query head) -- or a
// single tile at HD = 128, where tensor memory holds one tile's O -- sorted
// longest first; a persistent grid (one CTA per SM) walks them in snake
// order (CTA c takes items c, 2G-1-c, 2G+c, ...) so the causal work per CTA
// evens out.  Each K/V tile loaded serves both query tiles of an item.  At
// HD = 64, when pairs would leave SMs idle, the launch goes to
// prefill_split.cu instead (one query tile per item, its keys split between
// the two softmax warpgroups).
//  * warp 8, one thread: TMA (cp.async.bulk.tensor, 128-byte swizzle) loads
//    the Q tile(s) once and streams 128-key K and V tiles through a ring of
//    4 stages (d = 64) or 3 (d = 128).
//  * warp 9, one thread: issues tcgen05.mma (bf16 in, fp32 accumulate in
//    tensor memory) for S_A = Q_A K^T and S_B = Q_B K^T (128 TMEM columns
//    each) per K/V tile; warp 10, one thread: O_A += P_A V and O_B += P_B V,
//    with P read from tensor memory (64 columns of bf16 pairs per tile) and
//    O kept in tensor memory for the whole key loop.  Two issuing threads
//    took the 2048-token prefill from 28.9 to 24.9 us.  While one query
//    tile's softmax runs, the tensor core works on the other tile.  Warp 11
//    has no role.
//  * warps 0-3 (tile A) and 4-7 (tile B), thread r owns query row r (TMEM
//    lane quarter warp % 4): read the whole S row from TMEM into registers in
//    one round trip, mask the causal diagonal, find the row's largest scaled
//    score from the raw scores (their maximum, or their minimum for a
//    negative scale: the sign is a template parameter), keep the online
//    softmax in base 2 with one fused multiply-add per pair of exponents,
//    write P as bf16 pairs into tensor memory (tcgen05.st).  The running max
//    is raised only when a row's max grows by more than 2^8 (then O is
//    rescaled in TMEM); otherwise P may reach 2^8, harmless in fp32 sums and
//    bf16 P.  The softmax warpgroups take 208 registers per thread from the
//    issue warpgroup (setmaxnreg), which keeps the raw-score form free of
//    spills.
//  Scores never leave the SM (no S or P in HBM).
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace gqa {
namespace {

constexpr int kBM = 128;   // query rows per tile (MMA M)
constexpr int kBN = 128;   // keys per tile (MMA N of QK^T, K of PV)
constexpr int kQT = 2;     // query-tile slots per CTA (softmax warpgroups)
constexpr int kMaxKVStages = 4;
constexpr int kPThreads = 384;             // 12 warps
constexpr int kPTmaWarp = 8;               // TMA
constexpr int kPQKWarp = 9;                // QK^T issuer; allocates tensor memory
constexpr int kPVWarp = 10;                // the PV issuer
constexpr int kPRegsSoftmax = 208;
constexpr int kPRegsOther = 88;
constexpr int kPRegSplitTotal = 4 * 32 * (2 * kPRegsSoftmax + kPRegsOther);
static_assert(kPRegSplitTotal <= kPThreads * 168, "register split above the launch allocation");
constexpr int kChunkBytes = kBM * 64 * 2;  // 16 KB: 128 rows x 128 bytes, one swizzle column block
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemP = 256;           // P of tile x at 256 + 64x (bf16 pairs)
constexpr uint32_t kTmemO = 384;           // O of tile x at 384 + HD*x
constexpr float kLazyTau = 8.0f;           // keep a stale max up to 2^8 below

// Per head dim HD (64 or 128): a 128-row tile of HD bf16 is HD/64 column
// blocks of 128 bytes (the 128-byte swizzle span), each 16 KB, one after the
// other.  TMEM holds S (128 columns), P (64) and O (HD) per query tile: two
// tiles for HD=64 (S 0..255, P 256..383, O 384..511), one for HD=128
// (S 0..127, P 256..319, O 384..511).
template <int HD>
struct PL {
  static constexpr int kChunks = HD / 64;
  static constexpr int kTileBytes = kBM * HD * 2;
  static constexpr int kQTiles = HD == 64 ? 2 : 1;  // query tiles an item may hold
  static constexpr int kStages = HD == 64 ? 4 : 3;  // K/V ring depth
  // shared memory map (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;                                   // query tile x
  static constexpr int kOffKV = kOffQ + kQTiles * kTileBytes;       // stage s: K, then V
  static constexpr int kOffBar = kOffKV + kStages * 2 * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;           // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kTmemO + kQTiles * HD <= kTmemCols, "tensor memory columns");
};

// barrier slots
constexpr int kBarQ = 0;
constexpr int kBarKVFull = 1;                     // + stage
constexpr int kBarKVEmpty = kBarKVFull + kMaxKVStages;
constexpr int kBarSFull = kBarKVEmpty + kMaxKVStages;  // + tile
constexpr int kBarSFree = kBarSFull + kQT;
constexpr int kBarPFull = kBarSFree + kQT;    // + tile
constexpr int kBarPVDone = kBarPFull + kQT;   // + tile
constexpr int kBarOFree = kBarPVDone + kQT;   // + tile: epilogue has read O
constexpr int kBarQFree = kBarOFree + kQT;    // QK^T of the item has read Q
constexpr int kNumBars = kBarQFree + 1;

__device__ unsigned int g_prefill_timeouts;   // CTAs whose wait gave up; read by prefill_read_timeouts
__device__ unsigned int g_prefill_skips;      // debug builds: accesses a range check skipped

struct PrefillParams {
  uint16_t* out;
  int S, start_pos, Hq, Hkv, g;
  int tpi;      // query tiles per work item: 2, or 1 when pairs would not fill the SMs
  int n_units;  // work units per head: ceil(query tiles / tpi)
  float scale_log2;  // scale * log2(e)
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_wait(bar, parity, abort_flag)) return true;
  if (!*abort_flag) atomicAdd(&g_prefill_timeouts, 1u);
  *abort_flag = 1;
  return false;
}

// The same for a whole warp that goes on to warp-collective TMEM loads and
// stores (.sync.aligned): the outcome is made uniform over the warp, so
// either every lane carries on or every lane stops.
__device__ __forceinline__ bool warp_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
}

template <int HD, bool kPos>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  using L = PL<HD>;
  constexpr int kKVStages = L::kStages;
  constexpr int kTileBytes = L::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.n_units * p.Hq;
  const int G = gridDim.x;
  // Work item w (longest first): query-tile unit n_units-1-w/Hq of head w%Hq
  // (a unit is tpi consecutive 128-token query tiles).
  // CTA c takes items c, 2G-1-c, 2G+c, 4G-1-c, ... (a snake over the sorted
  // list), which evens out the causal work per CTA.
  auto item_of = [&](int r) -> int {
    return r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  };
  struct Item {
    int h, kvh, q0, nt[kQT], n;
  };
  auto item = [&](int w) -> Item {
    Item it;
    it.h = w % p.Hq;
    it.kvh = it.h / p.g;
    it.q0 = (p.n_units - 1 - w / p.Hq) * p.tpi * kBM;
    it.n = 0;
#pragma unroll
    for (int x = 0; x < kQT; ++x) {  // key tiles query tile x needs (0: no query rows)
      const int r0 = it.q0 + x * kBM;
      it.nt[x] = (x < p.tpi && r0 < p.S) ? (p.start_pos + min(r0 + kBM, p.S) + kBN - 1) / kBN : 0;
      it.n = max(it.n, it.nt[x]);
    }
    return it;
  };

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    mbar_init(bar(kBarQFree), 1);
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(bar(kBarKVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
    }
    for (int x = 0; x < kQT; ++x) {
      mbar_init(bar(kBarSFull + x), 1);
      mbar_init(bar(kBarSFree + x), 128);
      mbar_init(bar(kBarPFull + x), 128);
      mbar_init(bar(kBarPVDone + x), 1);
      mbar_init(bar(kBarOFree + x), 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kPQKWarp) {
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
  // Launched with programmatic stream serialisation: the set-up above may
  // run while the previous kernel on the stream finishes; q, k, v and out
  // are touched only after this wait.
  grid_dependency_wait();
  grid_dependents_launch();
  // TMEM columns: S of tile x [128x, +128); P of tile x [256+64x, +64);
  // O of tile x [384+64x, +64)
  const uint32_t sQ = base + L::kOffQ;
  // one 128-row tile: its HD/64 column blocks, each at +16 KB
  // (debug builds: a tile outside [0, heads) x [0, rows) is not loaded, and
  // the CTA stops)
  auto tma_tile = [&](uint32_t dst, const CUtensorMap* map, int head, int row, uint32_t b,
                      int heads, int rows) {
    if (!range_ok_count(head >= 0 && head < heads && row >= 0 && row < rows, &g_prefill_skips)) {
      *abort_flag = 1;
      return;
    }
#pragma unroll
    for (int c = 0; c < L::kChunks; ++c) tma_load_3d(dst + c * kChunkBytes, map, 64 * c, head, row, b);
  };

  // Every mbarrier completes one phase per use; parities below come from
  // running counts kept across this CTA's items.
  auto regs_down = [] { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPRegsOther)); };
  auto regs_up = [] { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPRegsSoftmax)); };
  if (warp == kPTmaWarp) {
    // ------------------------------------------------------ TMA producer --
    regs_down();
    if (lane == 0) {
      uint32_t gk = 0;  // K/V tiles issued so far
      for (int r = 0; item_of(r) < n_items; ++r) {
        const Item it = item(item_of(r));
        // the previous item's QK^T MMAs have finished reading Q
        if (r > 0 && !wait_or_abort(bar(kBarQFree), (uint32_t)(r - 1) & 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(kBarQ), p.tpi * kTileBytes);
        for (int x = 0; x < p.tpi; ++x)
          // a second tile past the last query row is loaded (zero fill) but unused
          tma_tile(sQ + x * kTileBytes, &tm_q, it.h, it.q0 + x * kBM, bar(kBarQ), p.Hq,
                   it.nt[x] > 0 ? p.S : p.S + kBM);
        bool ok = true;
        for (int i = 0; i < it.n; ++i, ++gk) {
          const int s = gk % kKVStages;
          const uint32_t u = gk / kKVStages;
          if (gk >= kKVStages && !wait_or_abort(bar(kBarKVEmpty + s), (u - 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t sK = base + L::kOffKV + s * 2 * kTileBytes;
          mbar_arrive_expect_tx(bar(kBarKVFull + s), 2 * kTileBytes);
          tma_tile(sK, &tm_k, it.kvh, i * kBN, bar(kBarKVFull + s), p.Hkv, p.start_pos + p.S);
          tma_tile(sK + kTileBytes, &tm_v, it.kvh, i * kBN, bar(kBarKVFull + s), p.Hkv,
                   p.start_pos + p.S);
        }
        if (!ok) break;
      }
    }
  } else if (warp == kPQKWarp) {
    // ----------------------------------------------- QK^T issuer (S_x) --
    regs_down();
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(kBM, kBN, false);
      uint32_t gk = 0;             // K/V tiles consumed so far
      uint32_t cs[kQT] = {0, 0};   // S_x issued so far
      bool ok = true;
      for (int r = 0; ok && item_of(r) < n_items; ++r) {
        const Item it = item(item_of(r));
        if (!wait_or_abort(bar(kBarQ), (uint32_t)r & 1u, abort_flag)) break;
        const uint32_t gk0 = gk;
        for (int i = 0; ok && i < it.n; ++i) {
          const uint32_t g = gk0 + i;
          const int s = g % kKVStages;
          if (!wait_or_abort(bar(kBarKVFull + s), (g / kKVStages) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t sK = base + L::kOffKV + s * 2 * kTileBytes;
          for (int x = 0; ok && x < kQT; ++x) {
            if (i >= it.nt[x]) continue;
            // the softmax has read the previous S_x
            if (cs[x] > 0 &&
                !wait_or_abort(bar(kBarSFree + x), (cs[x] - 1) & 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {  // 4 K-steps per 128-byte column block
              const uint32_t off = (k >> 2) * kChunkBytes + (k & 3) * 32;
              tc_mma(tmem + 128 * x, sw128_desc(sQ + x * kTileBytes + off), sw128_desc(sK + off),
                     idesc_qk, k > 0);
            }
            tc_commit(bar(kBarSFull + x));
            ++cs[x];
          }
          if (ok && i + 1 == it.n) tc_commit(bar(kBarQFree));  // last QK^T of this item
        }
        gk = gk0 + it.n;
      }
    }
  } else if (warp == kPVWarp) {
    // ------------------------------------------------ PV issuer (O_x) --
    // Its own thread, so that the two streams of MMAs are issued in
    // parallel.  P_x of tile j is written after S_x of tile j was read, so
    // the QK^T that read the stage's K is done once P_x is; the commit after
    // the tile's last PV therefore releases the whole stage.
    regs_down();
    if (lane == 0) {
      // O (+)= P V at N = HD: V's HD/64 column blocks, kChunkBytes apart
      constexpr uint32_t idesc_pv = make_idesc(kBM, HD, true);
      uint32_t gk = 0;             // K/V tiles consumed so far
      uint32_t cp[kQT] = {0, 0};   // P_x consumed (PV_x issued) so far
      bool ok = true;
      for (int r = 0; ok && item_of(r) < n_items; ++r) {
        const Item it = item(item_of(r));
        const uint32_t gk0 = gk;
        for (int j = 0; ok && j < it.n; ++j) {
          for (int x = 0; ok && x < kQT; ++x) {
            if (j >= it.nt[x]) continue;
            if (j == 0 && r > 0 &&  // the previous item's epilogue has read O_x
                !wait_or_abort(bar(kBarOFree + x), (uint32_t)(r - 1) & 1u, abort_flag)) {
              ok = false;
              break;
            }
            if (!wait_or_abort(bar(kBarPFull + x), cp[x] & 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sV =
                base + L::kOffKV + ((gk0 + j) % kKVStages) * 2 * kTileBytes + kTileBytes;
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k)
              tc_mma_ts(tmem + kTmemO + HD * x, tmem + kTmemP + 64 * x + 8 * k,
                        sw128_desc(sV + k * 16 * 128, HD > 64 ? kChunkBytes : 16), idesc_pv,
                        (j > 0 || k > 0) ? 1u : 0u);
            tc_commit(bar(kBarPVDone + x));
            ++cp[x];
          }
          if (ok) tc_commit(bar(kBarKVEmpty + (gk0 + j) % kKVStages));  // tile j released
        }
        gk = gk0 + it.n;
      }
    }
  } else if (warp > kPVWarp) {
    regs_down();  // warp 11: no role
  } else {
    // ------------------------------------------- softmax / epilogue (r) --
    regs_up();
    const int x = warp >> 2;                            // query tile of this warpgroup
    const int sub = warp & 3;                           // TMEM lane quarter
    const int r = sub * 32 + lane;                      // row within the tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t tm_S = tmem + 128 * x + lane_off;
    const uint32_t tm_O = tmem + kTmemO + HD * x + lane_off;
    const uint32_t tm_P = tmem + kTmemP + 64 * x + lane_off;
    const float c = p.scale_log2;  // non-zero (the host replaces 0 by a tiny value)
    constexpr bool c_pos = kPos;    // the scale's sign, a launch choice
    const float mask_raw = c_pos ? -INFINITY : INFINITY;  // times c: -inf
    uint32_t cs = 0;   // S_x consumed so far
    uint32_t cpv = 0;  // PV_x issued before this item
    bool ok = true;

    for (int rr = 0; ok && item_of(rr) < n_items; ++rr) {
      const Item it = item(item_of(rr));
      const int row = it.q0 + x * kBM + r;             // query token index
      const int qpos = p.start_pos + row;              // its absolute position
      const int nt = it.nt[x];
      float m_run = -INFINITY, l_run = 0.f;
      auto wait_pv = [&](int j) -> bool {  // PV_x of tile j of this item done
        if (!warp_wait_or_abort(bar(kBarPVDone + x), (cpv + j) & 1u, abort_flag)) return false;
        tc_fence_after();
        return true;
      };

      for (int i = 0; i < nt; ++i, ++cs) {
        if (!warp_wait_or_abort(bar(kBarSFull + x), cs & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const int kbase = i * kBN;
        const bool diag = kbase + kBN - 1 > qpos;

        // the whole S row in one round trip
        float sv[kBN];
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          float* dst = sv + cc * 32;
          tmem_ld32(tm_S + cc * 32, *reinterpret_cast<float(*)[32]>(dst));
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + x));       // S_x may be overwritten

        // The row's largest scaled score from the raw scores: their maximum
        // when the scale is positive, their minimum when it is negative (8
        // independent three-input chains), times c.  Masked keys (diagonal
        // tiles only) take the raw value that neither can pick.
        if (diag) {
#pragma unroll
          for (int j = 0; j < kBN; ++j) sv[j] = (kbase + j > qpos) ? mask_raw : sv[j];
        }
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = sv[a];
#pragma unroll
        for (int j = 8; j < kBN; j += 2)
          mx8[(j >> 1) & 7] = c_pos ? fmax3(mx8[(j >> 1) & 7], sv[j], sv[j + 1])
                                    : fmin3(mx8[(j >> 1) & 7], sv[j], sv[j + 1]);
        const float mr = c_pos ? fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]))
                               : fmin3(fmin3(mx8[0], mx8[1], mx8[2]), fmin3(mx8[3], mx8[4], mx8[5]),
                                       fminf(mx8[6], mx8[7]));
        const float mx = mr * c;

        // PV of tile i-1 done: O is stable and P_x may be overwritten
        if (i > 0 && !wait_pv(i - 1)) { ok = false; break; }
        // Raise the running max on the first tile, or when it grew by more
        // than 2^8.  The O rescale below uses warp-collective TMEM loads and
        // stores, so the decision is taken for the whole warp: rows whose
        // max did not grow keep it and scale by 1.
        const bool grow = mx > m_run + kLazyTau;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? ex2(m_run - mx) : 1.f;
          m_run = grow ? mx : m_run;
          l_run *= alpha;
          if (i > 0) {
#pragma unroll 1
            for (int cc = 0; cc < HD / 16; ++cc) {
              float o[16];
              tmem_ld16(tm_O + cc * 16, o);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] *= alpha;
              tmem_st16(tm_O + cc * 16, o);
            }
          }
        }

        // P = 2^(s*c - m) (exactly 0 where masked: 2^-inf) as bf16 pairs into
        // TMEM: column q of P holds keys 2q (low half) and 2q+1 (high half)
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        const f2 c2 = mk2(c, c);
        const f2 m2 = mk2(-m_use, -m_use);
        f2 rs2[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) rs2[a] = mk2(0.f, 0.f);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float pw[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int j = half * 64 + 2 * q;
            float lo, hi;
            brk2(fma2(mk2(sv[j], sv[j + 1]), c2, m2), lo, hi);
            lo = ex2(lo);
            hi = ex2(hi);
            rs2[q & 3] = add2(rs2[q & 3], mk2(lo, hi));
            pw[q] = __uint_as_float(pack_bf16x2(lo, hi));
          }
          tmem_st32(tm_P + half * 32, pw);
        }
        {
          f2 t = add2(add2(rs2[0], rs2[1]), add2(rs2[2], rs2[3]));
          float lo, hi;
          brk2(t, lo, hi);
          l_run += lo + hi;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + x));       // P_x (and any O rescale) ready
      }

      // epilogue: O / l for row r (128 contiguous bytes)
      if (ok && nt > 0) {
        ok = wait_pv(nt - 1);
        const float inv = ok ? 1.f / l_run : __int_as_float(0x7fc00000);
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)row * p.Hq + it.h) * HD);
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          float o[32];
          tmem_ld32(tm_O + cc * 32, o);
          tmem_ld_wait();
          if (row < p.S && range_ok_count(row >= 0 && it.h < p.Hq, &g_prefill_skips)) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              uint4 w;
              w.x = pack_bf16x2(o[q8 * 8 + 0] * inv, o[q8 * 8 + 1] * inv);
              w.y = pack_bf16x2(o[q8 * 8 + 2] * inv, o[q8 * 8 + 3] * inv);
              w.z = pack_bf16x2(o[q8 * 8 + 4] * inv, o[q8 * 8 + 5] * inv);
              w.w = pack_bf16x2(o[q8 * 8 + 6] * inv, o[q8 * 8 + 7] * inv);
              dst[cc * 4 + q8] = w;
            }
          }
        }
      }
      cpv += nt;
      tc_fence_before();
      mbar_arrive(bar(kBarOFree + x));  // O_x may be overwritten by the next item
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
  if (warp == kPQKWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host --

// [tokens, heads, hd] bf16 viewed as 3-D (hd, heads, tokens); box 64 x 1 x 128
// (one 128-byte column block of a tile; hd = 128 takes two boxes).
bool make_map(CUtensorMap* m, const void* ptr, int tokens, int heads, int hd) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)heads * hd * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int Hq, int Hkv, int d) {
  return (d == 64 || d == 128) && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && Hq <= 65535;
}

namespace {

template <int HD>
cudaError_t launch_prefill_hd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                              PrefillParams p, cudaStream_t stream) {
  using L = PL<HD>;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    for (auto kern : {prefill_tcgen05_kernel<HD, true>, prefill_tcgen05_kernel<HD, false>}) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           L::kSmemBytes);
      if (e != cudaSuccess) return e;
      // registers move between warpgroups (setmaxnreg): the launch
      // allocation must cover the split
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if ((long long)fa.numRegs * kPThreads < kPRegSplitTotal) return cudaErrorInvalidConfiguration;
    }
    configured[dev] = true;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  // Two query tiles per item share each K/V tile and keep both softmax
  // warpgroups busy.  When that leaves SMs idle at HD = 64, one tile per
  // item with its keys split between the two softmax warpgroups
  // (prefill_split.cu); at HD = 128, where tensor memory holds one tile's O,
  // one tile per item here.
  const long long n_qt = (p.S + kBM - 1) / kBM;
  if (HD == 64 && (n_qt + 1) / 2 * (long long)p.Hq < sms)
    return launch_prefill_split(mq, mk, mv, p.S, p.start_pos, p.Hq, p.Hkv, p.scale_log2, p.out,
                                sms, stream);
  p.tpi = L::kQTiles == 1 ? 1 : kQT;
  p.n_units = (int)((n_qt + p.tpi - 1) / p.tpi);
  const long long items = (long long)p.n_units * p.Hq;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)std::min<long long>(items, sms);  // one CTA per SM
  // programmatic dependent launch: the set-up overlaps the previous kernel
  auto kern =
      p.scale_log2 > 0.f ? prefill_tcgen05_kernel<HD, true> : prefill_tcgen05_kernel<HD, false>;
  return launch_pdl(kern, dim3(blocks), dim3(kPThreads), (size_t)L::kSmemBytes, stream, mq, mk, mv,
                    p);
}

}  // namespace

// The prefill waits that gave up since the last call (their kernels stopped
// early, so some output rows were not written); clears the count.
cudaError_t prefill_read_timeouts(uint32_t* count, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  unsigned v = 0, v_split = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_prefill_timeouts, sizeof(v));
  if (e == cudaSuccess && v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_prefill_timeouts, &zero, sizeof(zero));
  }
  if (e == cudaSuccess) e = prefill_split_read_timeouts(&v_split);
  *count = v + v_split;
  return e;
}

// Debug builds: the accesses a range check skipped since the last call (both
// prefill kernels); clears the count.  Always 0 in other builds.
cudaError_t prefill_read_skips(uint32_t* count, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  unsigned v = 0, v_split = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_prefill_skips, sizeof(v));
  if (e == cudaSuccess && v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_prefill_skips, &zero, sizeof(zero));
  }
  if (e == cudaSuccess) e = prefill_split_read_skips(&v_split);
  *count = v + v_split;
  return e;
}

cudaError_t launch_prefill(const void* q, const void* k, const void* v, int S, int start_pos,
                           int Hq, int Hkv, int d, float scale, void* out,
                           cudaStream_t stream) {
  const int T = start_pos + S;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, S, Hq, d) || !make_map(&mk, k, T, Hkv, d) ||
      !make_map(&mv, v, T, Hkv, d))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.out = static_cast<uint16_t*>(out);
  p.S = S;
  p.start_pos = start_pos;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (p.scale_log2 == 0.f) p.scale_log2 = 1e-30f;  // 2^(s*c - m) then rounds to exactly 1
  p.tpi = 1;
  p.n_units = 0;
  return d == 128 ? launch_prefill_hd<128>(mq, mk, mv, p, stream)
                  : launch_prefill_hd<64>(mq, mk, mv, p, stream);
}

}  // namespace gqa
