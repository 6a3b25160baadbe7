// prefill_split.cu -- causal prefill at head dim 64 for work items of one
// 128-token query tile: the two softmax warpgroups of a CTA split the item's
// key tiles between them and merge at the end (tcgen05 tensor cores).
//
// What it computes is what prefill.cu computes ("step14_3 -- batched
// attention", sections "problem" and "F.scaled_dot_product_attention";
// "MiniCPM4 `forward_step` Attention Performance Fix", section 5): token i of
// the S new ones (absolute position start_pos + i) attends keys
// 0..start_pos+i, query head h reads KV head h/g, out [S,Hq,64] bf16.
//
// When to use it: when two query tiles per work item would leave SMs idle
// (the 512-token chunk over a 2048-token prefix has 128 one-tile items for
// 152 SMs), prefill.cu's one-tile items keep one softmax warpgroup busy and
// the other idle, and each key tile's softmax waits on the P.V it has just
// issued (a group of 8 MMAs completes about 300 cycles after issue on this
// part).  Here both warpgroups ("lanes") work on the item's query tile, lane x
// taking the key tiles i with i % 2 == x, so one lane's exponentials overlap
// the other lane's MMAs; lane 0 merges the two partial results (max, sum,
// unnormalised O) at the end.  On the 512-over-2048 workload this took the
// launch from 26.7 to 22.6 us.
//
//  * warp 8, one thread: TMA (cp.async.bulk.tensor, 128-byte swizzle) loads
//    the item's query tile and streams 128-key K and V tiles through a
//    6-stage ring.
//  * warp 9 issues S_x = Q K_i^T (M = 128, N = 128, 4 x K16; fp32 in tensor
//    memory); warp 10 issues O_x += P_x V_i (A = P from tensor memory, B = V
//    from shared memory, N = 64).  Each runs its loop warp-uniformly and one
//    elected lane issues the MMAs and commits: an M=128, N=64 MMA with A in
//    tensor memory then issues at its tensor-core time of 32 cycles, against
//    46-49 cycles from a loop one thread runs alone in a divergent branch.
//  * warps 0-3 (lane 0) and 4-7 (lane 1), thread r owns query row r (TMEM
//    lane quarter warp % 4): read the S row from tensor memory in one round
//    trip, mask the causal diagonal, keep the online softmax in base 2 (the
//    running max raised only when it grows by more than 2^8), write P as
//    bf16 pairs into tensor memory.
//  Tensor memory per lane x: S (128 columns) at 128x, P (64 columns of bf16
//  pairs) at 256 + 64x, O (64) at 384 + 64x.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace gqa {
namespace {

constexpr int kHD = 64;
constexpr int kBM = 128;   // query rows per tile (MMA M)
constexpr int kBN = 128;   // keys per tile (MMA N of QK^T, K of PV)
constexpr int kLanes = 2;  // softmax warpgroups
constexpr int kStages = 6; // K/V ring depth
constexpr int kThreads = 384;  // 12 warps
constexpr int kTmaWarp = 8;
constexpr int kQKWarp = 9;     // S issuer; allocates tensor memory
constexpr int kPVWarp = 10;    // O issuer
constexpr int kTileBytes = kBM * kHD * 2;  // 16 KB: 128 rows x 128 bytes, one swizzle span
constexpr uint32_t kTmemCols = 512;
constexpr float kLazyTau = 8.0f;           // keep a stale max up to 2^8 below
// Registers per thread after the prologue: the two softmax warpgroups hold a
// whole 128-key S row each, the third (TMA and MMA issue) needs few.  The
// split must fit the block's launch allocation (kThreads x the kernel's
// register count, at most 168 at this block size); the host checks that
// before every launch, since a larger split would wait for ever.
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 88;
constexpr int kRegSplitTotal = 4 * 32 * (kLanes * kRegsSoftmax + kRegsOther);
static_assert(kRegSplitTotal <= kThreads * 168, "register split above the launch allocation");

constexpr uint32_t tmS(int x) { return 128u * x; }
constexpr uint32_t tmP(int x) { return 256u + 64u * x; }
constexpr uint32_t tmO(int x) { return 384u + 64u * x; }

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kTileBytes;                  // stage s: K, then V
constexpr int kOffML = kOffKV + kStages * 2 * kTileBytes;   // lane 1's (max, sum) per row
constexpr int kOffBar = kOffML + kBM * 8;
constexpr int kSmemBytes = kOffBar + 256 + 1024;            // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// barrier slots
constexpr int kBarQ = 0;
constexpr int kBarKVFull = 1;                          // + stage
constexpr int kBarKVEmpty = kBarKVFull + kStages;
constexpr int kBarSFull = kBarKVEmpty + kStages;       // + lane
constexpr int kBarSFree = kBarSFull + kLanes;
constexpr int kBarPFull = kBarSFree + kLanes;
constexpr int kBarPVDone = kBarPFull + kLanes;
constexpr int kBarOFree = kBarPVDone + kLanes;         // + lane: lane 0 has read O_x
constexpr int kBarQFree = kBarOFree + kLanes;          // the item's QK^T have read Q
constexpr int kBarMerge = kBarQFree + 1;               // lane 1's (max, sum) are in shared memory
constexpr int kNumBars = kBarMerge + 1;

__device__ unsigned int g_split_timeouts;  // CTAs whose wait gave up
__device__ unsigned int g_split_skips;     // debug builds: accesses a range check skipped

struct SplitParams {
  uint16_t* out;
  int S, start_pos, Hq, Hkv, g;
  int n_qt;          // query tiles per head
  float scale_log2;  // scale * log2(e), never 0
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_wait(bar, parity, abort_flag)) return true;
  if (!*abort_flag) atomicAdd(&g_split_timeouts, 1u);
  *abort_flag = 1;
  return false;
}

// The same for a whole warp (warp-uniform loops, warp-collective TMEM loads
// and stores): the outcome is made uniform over the warp, so either every
// lane carries on or every lane stops.
__device__ __forceinline__ bool warp_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
}

// One work item: query tile starting at row q0 of head h; n key tiles, lane x
// taking tiles x, x + 2, ...
struct Item {
  int h, kvh, q0, n;
  __device__ __forceinline__ int units(int x) const { return x == 0 ? (n + 1) >> 1 : n >> 1; }
};

template <bool kPos>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float2* lane1_ml = reinterpret_cast<float2*>(smem + kOffML);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.n_qt * p.Hq;
  const int G = gridDim.x;
  // Work item w (longest first): query tile n_qt-1-w/Hq of head w%Hq.  CTA c
  // takes items c, 2G-1-c, 2G+c, 4G-1-c, ... (a snake over the sorted list),
  // which evens out the causal work per CTA.
  auto item_of = [&](int r) -> int {
    return r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  };
  auto item = [&](int w) -> Item {
    Item it;
    it.h = w % p.Hq;
    it.kvh = it.h / p.g;
    it.q0 = (p.n_qt - 1 - w / p.Hq) * kBM;
    it.n = (p.start_pos + min(it.q0 + kBM, p.S) + kBN - 1) / kBN;
    return it;
  };

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarMerge), 128);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
    }
    for (int x = 0; x < kLanes; ++x) {
      mbar_init(bar(kBarSFull + x), 1);
      mbar_init(bar(kBarSFree + x), 128);
      mbar_init(bar(kBarPFull + x), 128);
      mbar_init(bar(kBarPVDone + x), 1);
      mbar_init(bar(kBarOFree + x), 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kQKWarp) {
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
  const uint32_t sQ = base + kOffQ;

  // Registers move from the issue warpgroup (warps 8-11) to the two softmax
  // warpgroups: every warp of a warpgroup runs the same setmaxnreg, first
  // thing in its role's branch, before any wait.
  auto regs_down = [] { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther)); };
  auto regs_up = [] { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax)); };

  // Every mbarrier completes one phase per use; parities below come from
  // running counts kept across this CTA's items.
  if (warp == kTmaWarp) {
    // ------------------------------------------------------ TMA producer --
    regs_down();
    if (lane == 0) {
      uint32_t gk = 0;  // K/V tiles issued so far
      for (int r = 0; item_of(r) < n_items; ++r) {
        const Item it = item(item_of(r));
        // the previous item's QK^T MMAs have finished reading Q
        if (r > 0 && !wait_or_abort(bar(kBarQFree), (uint32_t)(r - 1) & 1u, abort_flag)) break;
        // (debug builds: a tile outside the query, key or value rows is not
        // loaded, and the CTA stops)
        if (!range_ok_count(it.h >= 0 && it.h < p.Hq && it.q0 >= 0 && it.q0 < p.S &&
                                it.kvh >= 0 && it.kvh < p.Hkv &&
                                (it.n - 1) * kBN < p.start_pos + p.S,
                            &g_split_skips)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarQ), kTileBytes);
        tma_load_3d(sQ, &tm_q, 0, it.h, it.q0, bar(kBarQ));
        bool ok = true;
        for (int i = 0; i < it.n; ++i, ++gk) {
          const int s = gk % kStages;
          const uint32_t u = gk / kStages;
          if (gk >= kStages && !wait_or_abort(bar(kBarKVEmpty + s), (u - 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t sK = base + kOffKV + s * 2 * kTileBytes;
          mbar_arrive_expect_tx(bar(kBarKVFull + s), 2 * kTileBytes);
          tma_load_3d(sK, &tm_k, 0, it.kvh, i * kBN, bar(kBarKVFull + s));
          tma_load_3d(sK + kTileBytes, &tm_v, 0, it.kvh, i * kBN, bar(kBarKVFull + s));
        }
        if (!ok) break;
      }
    }
  } else if (warp == kQKWarp) {
    // ----------------------------------------------- QK^T issuer (S_x) --
    // The whole warp runs the issue loop (warp-uniform waits and
    // descriptors); the elected lane issues the MMAs and commits.
    regs_down();
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_qk = make_idesc(kBM, kBN, false);
    uint32_t gk = 0;                 // K/V tiles consumed so far
    uint32_t cs[kLanes] = {0, 0};    // S_x issued so far
    bool ok = true;
    for (int r = 0; ok && item_of(r) < n_items; ++r) {
      const Item it = item(item_of(r));
      if (!warp_wait_or_abort(bar(kBarQ), (uint32_t)r & 1u, abort_flag)) break;
      for (int i = 0; ok && i < it.n; ++i) {
        const uint32_t g = gk + i;
        const int s = g % kStages;
        const int x = i & 1;
        if (!warp_wait_or_abort(bar(kBarKVFull + s), (g / kStages) & 1u, abort_flag) ||
            // the softmax has read the previous S_x
            (cs[x] > 0 && !warp_wait_or_abort(bar(kBarSFree + x), (cs[x] - 1) & 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sK = base + kOffKV + s * 2 * kTileBytes;
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k)  // 4 K-steps of one 128-byte swizzle span
          tc_mma_by(leader, tmem + tmS(x), sw128_desc(sQ + k * 32), sw128_desc(sK + k * 32),
                    idesc_qk, k > 0);
        tc_commit_by(leader, bar(kBarSFull + x));
        ++cs[x];
        if (i + 1 == it.n) tc_commit_by(leader, bar(kBarQFree));  // last QK^T of this item
      }
      gk += it.n;
    }
  } else if (warp == kPVWarp) {
    // ------------------------------------------------ PV issuer (O_x) --
    // P_x of tile i is written after S_x of tile i was read, so the QK^T
    // that read the stage's K is done once P_x is; the commit after the
    // tile's P.V therefore releases the whole stage.
    regs_down();
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_pv = make_idesc(kBM, kHD, true);  // B = V, MN-major
    uint32_t gk = 0;                 // K/V tiles consumed so far
    uint32_t cp[kLanes] = {0, 0};    // P_x consumed (PV_x issued) so far
    bool ok = true;
    for (int r = 0; ok && item_of(r) < n_items; ++r) {
      const Item it = item(item_of(r));
      for (int i = 0; ok && i < it.n; ++i) {
        const int x = i & 1;
        const bool first = i < 2;  // the lane's first tile of this item
        if ((first && r > 0 &&  // lane 0 has read the previous item's O_x
             !warp_wait_or_abort(bar(kBarOFree + x), (uint32_t)(r - 1) & 1u, abort_flag)) ||
            !warp_wait_or_abort(bar(kBarPFull + x), cp[x] & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sV = base + kOffKV + ((gk + i) % kStages) * 2 * kTileBytes + kTileBytes;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          tc_mma_ts_by(leader, tmem + tmO(x), tmem + tmP(x) + 8 * k,
                       sw128_desc(sV + k * 16 * 128), idesc_pv, (!first || k > 0) ? 1u : 0u);
        tc_commit_by(leader, bar(kBarPVDone + x));
        tc_commit_by(leader, bar(kBarKVEmpty + (gk + i) % kStages));  // tile i released
        ++cp[x];
      }
      gk += it.n;
    }
  } else if (warp >= 4 * kLanes) {
    regs_down();  // warp 11: no role
  } else {
    // ------------------------------------------- softmax / epilogue (r) --
    regs_up();
    const int x = warp >> 2;                            // lane of this warpgroup
    const int sub = warp & 3;                           // TMEM lane quarter
    const int r = sub * 32 + lane;                      // row within the tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t tm_S = tmem + tmS(x) + lane_off;
    const uint32_t tm_P = tmem + tmP(x) + lane_off;
    const uint32_t tm_O = tmem + tmO(x) + lane_off;
    const float c = p.scale_log2;  // non-zero (the host replaces 0 by a tiny value)
    constexpr bool c_pos = kPos;  // the scale's sign, a launch choice
    const float mask_raw = c_pos ? -INFINITY : INFINITY;  // times c: -inf
    uint32_t cs = 0;   // S_x consumed so far (= P_x written = PV_x issued)
    bool ok = true;

    for (int rr = 0; ok && item_of(rr) < n_items; ++rr) {
      const Item it = item(item_of(rr));
      const int row = it.q0 + r;                // query token index
      const int qpos = p.start_pos + row;       // its absolute position
      const int nx = it.units(x);
      float m_run = -INFINITY, l_run = 0.f;
      auto wait_pv = [&](uint32_t unit) -> bool {  // PV_x of the lane's unit-th tile done
        if (!warp_wait_or_abort(bar(kBarPVDone + x), unit & 1u, abort_flag)) return false;
        tc_fence_after();
        return true;
      };

      for (int i = x, j = 0; ok && i < it.n; i += 2, ++j) {
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

        // The row's largest scaled score, found on the raw scores: their
        // maximum when the scale is positive, their minimum when it is
        // negative (8 independent three-input chains), times c.  Masked
        // keys (diagonal tiles only) take the value that neither can pick.
        if (diag) {
#pragma unroll
          for (int jj = 0; jj < kBN; ++jj) sv[jj] = (kbase + jj > qpos) ? mask_raw : sv[jj];
        }
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = sv[a];
        if (c_pos) {
#pragma unroll
          for (int jj = 8; jj < kBN; jj += 2)
            mx8[(jj >> 1) & 7] = fmax3(mx8[(jj >> 1) & 7], sv[jj], sv[jj + 1]);
        } else {
#pragma unroll
          for (int jj = 8; jj < kBN; jj += 2)
            mx8[(jj >> 1) & 7] = fmin3(mx8[(jj >> 1) & 7], sv[jj], sv[jj + 1]);
        }
        const float mr = c_pos ? fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]))
                               : fmin3(fmin3(mx8[0], mx8[1], mx8[2]), fmin3(mx8[3], mx8[4], mx8[5]),
                                       fminf(mx8[6], mx8[7]));
        const float mx = mr * c;  // -inf when every key of the tile is masked for this row

        // The previous P.V of this lane is done: O_x is stable and P_x may be
        // overwritten.
        if (j > 0 && !wait_pv(cs - 1)) { ok = false; break; }
        // Raise the running max on the first visible key, or when it grew by
        // more than 2^8.  The O rescale below uses warp-collective TMEM loads
        // and stores, so the decision is taken for the whole warp: rows whose
        // max did not grow keep it and scale by 1.
        const bool grow = mx > m_run + kLazyTau;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? ex2(m_run - mx) : 1.f;  // m_run = -inf: 0
          m_run = grow ? mx : m_run;
          l_run *= alpha;
          if (j > 0) {
#pragma unroll 1
            for (int cc = 0; cc < kHD / 16; ++cc) {
              float o[16];
              tmem_ld16(tm_O + cc * 16, o);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) o[jj] *= alpha;
              tmem_st16(tm_O + cc * 16, o);
            }
          }
        }

        // P = 2^(s*c - m), one fused multiply-add per pair of keys (exactly
        // 0 where masked: the masked raw value times c is -inf), as bf16
        // pairs into TMEM: column q of P holds keys 2q (low half) and 2q+1
        // (high half).  A row that has seen no visible key yet (m = -inf:
        // lane 1's first tiles can lie wholly past it) takes m = 0, so its
        // masked keys give 2^-inf = 0 and not NaN.
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        const f2 c2 = mk2(c, c);
        const f2 m2 = mk2(-m_use, -m_use);
        f2 rs2[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) rs2[a] = mk2(0.f, 0.f);
#pragma unroll
        for (int qt = 0; qt < 4; ++qt) {
          float pw[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int jj = qt * 32 + 2 * q;
            float lo, hi;
            brk2(fma2(mk2(sv[jj], sv[jj + 1]), c2, m2), lo, hi);
            lo = ex2(lo);
            hi = ex2(hi);
            rs2[q & 3] = add2(rs2[q & 3], mk2(lo, hi));
            pw[q] = __uint_as_float(pack_bf16x2(lo, hi));
          }
          tmem_st16(tm_P + qt * 16, pw);
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
        ++cs;
      }

      // ---- epilogue: lane 1 hands over (max, sum), lane 0 merges ----
      // O_x of the lane's last tile is final once its P.V is done
      if (ok && nx > 0) ok = wait_pv(cs - 1);
      if (x == 1) {
        // (max, sum) of row r go to lane 0 once lane 0 has merged the
        // previous item's (it arrives on OFree_1 after reading them)
        if (rr > 0) ok = ok && warp_wait_or_abort(bar(kBarOFree + 1), (uint32_t)(rr - 1) & 1u,
                                                  abort_flag);
        lane1_ml[r] = make_float2(m_run, l_run);
        tc_fence_before();
        mbar_arrive(bar(kBarMerge));
      } else {
        // out = (a0 O0 + a1 O1) / (a0 l0 + a1 l1), a_x = 2^(m_x - max(m0, m1))
        ok = ok && warp_wait_or_abort(bar(kBarMerge), (uint32_t)rr & 1u, abort_flag);
        tc_fence_after();
        const float2 ml1 = lane1_ml[r];
        const bool has1 = it.units(1) > 0;  // O_1 holds this item's result
        const float M = fmaxf(m_run, ml1.x);
        const float a0 = ex2(m_run - M);
        const float a1 = has1 ? ex2(ml1.x - M) : 0.f;
        const float inv = 1.f / (a0 * l_run + a1 * ml1.y);
        const float w0 = a0 * inv, w1 = a1 * inv;
        const uint32_t tm_O1 = tmem + tmO(1) + lane_off;
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)row * p.Hq + it.h) * kHD);
        if (ok) {
#pragma unroll 1
          for (int cc = 0; cc < kHD / 32; ++cc) {
            float o[32], o1[32];
            tmem_ld32(tm_O + cc * 32, o);
            if (has1) tmem_ld32(tm_O1 + cc * 32, o1);
            tmem_ld_wait();
            if (!has1) {
#pragma unroll
              for (int q = 0; q < 32; ++q) o1[q] = 0.f;
            }
            if (row < p.S && range_ok_count(row >= 0 && it.h < p.Hq, &g_split_skips)) {
#pragma unroll
              for (int q8 = 0; q8 < 4; ++q8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = o[q8 * 8 + e] * w0 + o1[q8 * 8 + e] * w1;
                uint4 w;
                w.x = pack_bf16x2(v[0], v[1]);
                w.y = pack_bf16x2(v[2], v[3]);
                w.z = pack_bf16x2(v[4], v[5]);
                w.w = pack_bf16x2(v[6], v[7]);
                dst[cc * 4 + q8] = w;
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar(kBarOFree + 0));  // O_0 and O_1 may be overwritten by the next item,
        mbar_arrive(bar(kBarOFree + 1));  // and lane 1 may write its next (max, sum)
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
  if (warp == kQKWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_prefill_split(const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int S, int start_pos, int Hq, int Hkv,
                                 float scale_log2, void* out, int sms, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    for (auto kern : {prefill_split_kernel<true>, prefill_split_kernel<false>}) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
      if (e != cudaSuccess) return e;
      // The kernel moves registers between its warpgroups (setmaxnreg); the
      // block's launch allocation must cover the new split, or the softmax
      // warpgroups would wait for registers for ever.
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if ((long long)fa.numRegs * kThreads < kRegSplitTotal) return cudaErrorInvalidConfiguration;
    }
    configured[dev] = true;
  }
  SplitParams p;
  p.out = static_cast<uint16_t*>(out);
  p.S = S;
  p.start_pos = start_pos;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.n_qt = (S + kBM - 1) / kBM;
  p.scale_log2 = scale_log2 == 0.f ? 1e-30f : scale_log2;
  const long long items = (long long)p.n_qt * Hq;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)std::min<long long>(items, sms);  // one CTA per SM
  // programmatic dependent launch: the set-up overlaps the previous kernel
  auto kern = p.scale_log2 > 0.f ? prefill_split_kernel<true> : prefill_split_kernel<false>;
  return launch_pdl(kern, dim3(blocks), dim3(kThreads), (size_t)kSmemBytes, stream, mq, mk, mv, p);
}

cudaError_t prefill_split_read_timeouts(uint32_t* count) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_split_timeouts, sizeof(v));
  if (e == cudaSuccess && v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_split_timeouts, &zero, sizeof(zero));
  }
  *count = v;
  return e;
}

cudaError_t prefill_split_read_skips(uint32_t* count) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_split_skips, sizeof(v));
  if (e == cudaSuccess && v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_split_skips, &zero, sizeof(zero));
  }
  *count = v;
  return e;
}

}  // namespace gqa
