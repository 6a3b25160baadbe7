// decode_kernels.cuh -- split-KV decode attention over a static KV cache with
// GQA on CUDA cores, for group sizes g = 1, 2, 4: the kernels and their
// launch, included by one translation unit per group size (decode_g1.cu ...
// decode_g4.cu).  g = 8 runs on the tensor cores (decode_tc.cuh, which also
// uses the segment walk, helpers and merges defined here).
//
// What it computes ("MiniCPM4 `forward_step` Attention Performance Fix",
// sections 3 and 4.1): for every sequence b and query head h,
//   out[b,h,:] = softmax_j(scale * q[b,h,:] . K[b,h/g,j,:]) V[b,h/g,j,:]
// over cache rows j = 0..positions[b] only, or the last W of them with a
// local window (the slice replaces the
// full-length boolean mask of section 2.1, so the work follows position+1 and
// not max_len, sections 2.4 and 6.4).  Optionally the step's new K/V row is
// appended in the same launch (the page writes the row, then attends), and
// optionally q and the new key row are first rotated by the rotary embedding
// at each sequence's position (the page's apply_rotary_pos_emb, run before
// the cache write; rotate-half form, fp32, one rounding per operation), and
// optionally every position is advanced by one once the step has read them
// (a streaming step a CUDA graph can replay).  Rotation and advance are
// template flags, so the plain kernels carry neither.
//
// How (GB300 design, not the page's: the page calls PyTorch SDPA):
//  * The attended rows of every (sequence, KV head) pair -- a "segment" -- are
//    cut into 128-row tiles, streamed with 1-D bulk copies (TMA) into a
//    2-stage shared-memory ring guarded by mbarriers (128 KB in flight per
//    SM) by a producer warp (one thread).  Each tile is read from HBM once
//    and serves all g query heads of its KV head.
//  * 8 consumer warps (16 for g=1) each take 16 (8) keys of a tile; a key's
//    128 dims are spread over 16 lanes, 8 each, as fp32 pairs for the packed
//    fma.rn.f32x2.  q.k partial sums of the g heads are reduced across the
//    16 lanes with a transposing butterfly (each shuffle step halves the
//    number of heads still carried), and the softmax is kept
//    online in fp32 (running max and sum per head, in base 2 with
//    scale*log2(e) folded into q).
//  * Two ways to split a segment over CTAs, both computed on the device from
//    `positions` (one launch serves any positions; graph-capturable):
//    - cluster mode (few segments, e.g. B=1): one thread-block cluster of C
//      CTAs (8..16; the largest size that lets every
//      segment's cluster be resident at once) per segment; CTA rank r takes
//      tiles [r*n/C, (r+1)*n/C).  Each CTA stores its partial (max, sum,
//      unnormalised o) straight into rank 0's shared memory (distributed
//      shared memory); after one cluster barrier rank 0 merges them locally
//      -- no global scratch, no atomics.
//    - stream-K mode (many segments): all tiles of all segments form one flat
//      list; CTA c of a persistent grid (one per SM) takes
//      [c*T/G, (c+1)*T/G), balanced to one tile however ragged the batch is.
//      A segment split over CTAs is merged by the CTA that arrives last at
//      the segment's arrival counter (fp32 partials in the workspace; no
//      spin-wait).
#pragma once

#include <cfloat>
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "decode_params.h"

namespace gqa {
namespace {

namespace cg = cooperative_groups;

constexpr int kD = kDecodeD;
constexpr int kTile = 128;                         // keys per pipeline stage
constexpr int kStages = 2;
constexpr int kRowBytes = kD * 2;
constexpr int kTileBytes = kTile * kRowBytes;      // 32 KB per operand
constexpr int kMaxB = kDecodeMaxB;
constexpr int kMaxGrid = kDecodeMaxGrid;
constexpr int kMiscInts = 32;                      // [0] abort [1] last [8..8+NW) scan
constexpr int kWholeTiles = 4;                     // segments this short are not split
constexpr int kMaxCluster = 16;                    // CTAs per cluster in cluster mode

using Params = DecodeParams;

// Kernel variants: a mode M of compile-time flags, so that a plain step's
// kernel carries none of the optional work (even unused code moved register
// allocation and cost a few percent).
constexpr int kModeRope = 1;     // rotary embedding of q and the new key
constexpr int kModeAdvance = 2;  // positions += 1 after the step
constexpr int kModeWindow = 4;   // attend only the last p.window rows
constexpr int kModeMulti = 8;    // p.S new tokens per sequence (see head_row)

// Multi-token decode: the kernel's G "heads" of a KV head are p.S new tokens
// x g query heads (h = t*g + j), q and out are [B, S, Hq, D], token t sits at
// positions[b] + t and attends rows up to there.  Row of q/out for head h:
template <int G, bool MT>
__device__ __forceinline__ size_t head_row(const DecodeParams& p, int b, int kvh, int h) {
  if (!MT) return (size_t)b * p.Hq + (size_t)kvh * G + h;
  // g = G / S query heads per token, a power of two: token h >> log2(g)
  const int lg = 31 - __clz(G / p.S);
  const int gr = 1 << lg;
  return ((size_t)b * p.S + (h >> lg)) * p.Hq + (size_t)(kvh << lg) + (h & (gr - 1));
}

// Lanes per key (LPK): a key's 128 dims are spread over LPK lanes of a warp
// (128/LPK dims each), so a warp takes 32/LPK keys per step.  Fewer lanes
// per key means fewer shuffle-reduction steps but more q and o registers
// (128*g/LPK each).  16 lanes for every g: with 8, g = 4 ran at the
// register cap and spilled in its key loop (12% slower on the ragged batch),
// and g = 1 and 2 gained nothing from the shorter reduction either.
// These CUDA-core kernels serve g <= 4; g = 8 runs on the tensor cores
// (decode_tc.cuh), where its FMA work becomes two small MMAs per tile.
template <int G> struct Cfg {
  static_assert(G == 1 || G == 2 || G == 4, "the CUDA-core decode serves g <= 4");
  static constexpr int LPK = 16;
  static constexpr int NW = (G == 1) ? 16 : 8;
  // largest cluster: rank 0 keeps a landing slot for every rank's partial
  // (G x (kD + 2) floats each)
  static constexpr int kMaxC = 16;
  static constexpr int kThreads = (NW + 1) * 32;  // + the producer warp
  static constexpr int kConsumers = NW * 32;
  static constexpr int kKeysPerWarp = kTile / NW;  // 16 or 8
  static constexpr int kKeysPerStep = 32 / LPK;    // 2
  static constexpr int kIters = kKeysPerWarp / kKeysPerStep;
  // registers per thread that still let one CTA of kThreads fit the SM
  // (the register file is handed out as if the block were a multiple of
  // 128 threads)
  static constexpr int kRegsFit = 65536 / ((kThreads + 127) / 128 * 128);
  static constexpr int kMaxRegs = (kRegsFit > 255 ? 255 : kRegsFit) & ~7;
};

// A named barrier among the consumers, only for the one place every consumer
// warp reaches unconditionally: before the first tile wait.
template <int NC>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
}

// Barrier among the NW consumer warps everywhere else.  It sits on an
// mbarrier (count NW, one arrival per warp from lane 0 once the warp's lanes
// have synced) so that its wait is bounded like every other: a named barrier
// has no time limit, and a warp that gave up on a tile after a timeout would
// leave the others waiting at one for ever.
struct ConsumerSync {
  uint32_t bar;
  volatile int* abort_flag;
  uint32_t* status;
  uint32_t n;  // completed phases
  __device__ __forceinline__ void operator()(int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    if (!mbar_wait(bar, n & 1u, abort_flag) && lane == 0) {
      *abort_flag = 1;
      set_status(status, ATTN_DEV_TIMEOUT);
    }
    ++n;
    __syncwarp();
  }
};

// Position of flat tile t within (sequence, KV head, tile) order.
// Rows a step at position pos attends: n rows from lo (lo = 0 without a
// local window; with window W the last W rows, the current one included).
__device__ __forceinline__ void attended_rows(int pos, int window, int& lo, int& n) {
  lo = (window > 0 && pos >= window) ? pos - window + 1 : 0;
  n = pos - lo + 1;
}

struct Walk {
  int b, kvh, k, ntiles, n, lo;  // n attended rows of sequence b, from row lo
};

__device__ __forceinline__ void walk_init(Walk& w, long long t, const int* prefix,
                                          const int32_t* positions, int B, int Hkv, int window,
                                          int shift) {
  int lo = 0, hi = B - 1;  // largest b with Hkv*prefix[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)Hkv * prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  w.b = lo;
  w.ntiles = prefix[lo + 1] - prefix[lo];
  const long long off = t - (long long)Hkv * prefix[lo];
  w.kvh = (int)(off / w.ntiles);
  w.k = (int)(off % w.ntiles);
  attended_rows(positions[lo] + shift, window, w.lo, w.n);
}

__device__ __forceinline__ void walk_next(Walk& w, const int* prefix, const int32_t* positions,
                                          int B, int Hkv, int window, int shift) {
  if (++w.k < w.ntiles) return;
  w.k = 0;
  if (++w.kvh < Hkv) return;
  w.kvh = 0;
  do { ++w.b; } while (w.b < B && prefix[w.b + 1] == prefix[w.b]);
  if (w.b < B) {
    w.ntiles = prefix[w.b + 1] - prefix[w.b];
    attended_rows(positions[w.b] + shift, window, w.lo, w.n);
  }
}

// CTA whose tile range [c*T/G, (c+1)*T/G) contains flat tile t.
__device__ __forceinline__ int cta_of(long long t, long long T, int G) {
  return (int)(((unsigned long long)(t + 1) * G + T - 1) / T) - 1;
}

template <int G> struct Log2;
template <> struct Log2<1> { static constexpr int v = 0; };
template <> struct Log2<2> { static constexpr int v = 1; };
template <> struct Log2<4> { static constexpr int v = 2; };
template <> struct Log2<8> { static constexpr int v = 3; };
template <> struct Log2<16> { static constexpr int v = 4; };
template <> struct Log2<32> { static constexpr int v = 5; };

// Sum of acc[h] over the LPK lanes holding one key, for every head at once.
// A step with offset `off` keeps half of the heads and ships the other half
// to the partner lane, so after log2(G) steps each lane carries one head:
// head = lk >> (log2 LPK - log2 G).  The remaining steps are a plain butterfly.
template <int G, int LPK>
__device__ __forceinline__ float reduce_key(float (&acc)[G], int lk) {
  constexpr int LG = Log2<G>::v;
#pragma unroll
  for (int st = 0; st < LG; ++st) {
    const int off = (LPK / 2) >> st;
    const int n = G >> (st + 1);
    const bool upper = (lk & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = upper ? acc[n + i] : acc[i];
      const float send = upper ? acc[i] : acc[n + i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float v = acc[0];
#pragma unroll
  for (int off = (LPK / 2) >> LG; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// 8 bf16 (one 16-byte vector) -> 4 fp32 pairs (dims 2i, 2i+1).
__device__ __forceinline__ void unpack8x2(const uint4& u, f2 (&f)[4]) {
  f[0] = mk2(bf16lo(u.x), bf16hi(u.x));
  f[1] = mk2(bf16lo(u.y), bf16hi(u.y));
  f[2] = mk2(bf16lo(u.z), bf16hi(u.z));
  f[3] = mk2(bf16lo(u.w), bf16hi(u.w));
}

// Rotary embedding, rotate-half form, on N consecutive dims x of a row whose
// partner dims (64 away) are y: x' = x*cos + r*sin with r = -y in the first
// half of the row and r = y in the second.  Each product and the sum are
// rounded separately (no contraction into a fused multiply-add), so the
// result is the same fp32 value however the caller splits the row.
__device__ __forceinline__ float rope1(float x, float partner, float c, float sn,
                                       bool first_half) {
  const float r = first_half ? -partner : partner;
  return __fadd_rn(__fmul_rn(x, c), __fmul_rn(r, sn));
}

// Per-warp consumer state and math: one KV head's g query heads.  Lane
// `lane` works on key group grp = lane / LPK (32/LPK keys per step) and holds
// 128/LPK dims of that key: VPL 16-byte vectors, vector v covering dims
// 8*(lk + LPK*v) .. +8 (lk = lane % LPK), as fp32 pairs for fma.rn.f32x2.
template <int G>
struct Consumer {
  static constexpr int LG = Log2<G>::v;
  static constexpr int LPK = Cfg<G>::LPK;
  static constexpr int LL = Log2<LPK>::v;
  static constexpr int VPL = 16 / LPK;             // 16-byte vectors per lane per row
  static constexpr int NP = 4 * VPL;               // fp32 pairs per lane per row
  static constexpr int KPS = Cfg<G>::kKeysPerStep;
  static constexpr int KPW = Cfg<G>::kKeysPerWarp;
  static constexpr int IT = Cfg<G>::kIters;
  static constexpr float kTau = 8.0f;  // a stale running max may lag by 2^8
  f2 qf[G][NP];  // q[h][lane dims], pre-scaled by scale*log2(e)
  f2 o[G][NP];   // unnormalised output accumulators, same layout
  float m_run, l_run;  // for head hd (the same in every key group)
  int grp, lk, hd;
  int head_last;       // multi-token decode: last row head hd's token may see

  __device__ __forceinline__ void init(int lane) {
    grp = lane >> LL;
    lk = lane & (LPK - 1);
    hd = lk >> (LL - LG);  // head whose score this lane ends up with
  }
  __device__ __forceinline__ int dim_off(int v) const { return (lk + LPK * v) * 16; }  // bytes
  // the G query rows of KV head kvh of sequence b (head_row)
  template <bool MT>
  __device__ __forceinline__ void load_q(const DecodeParams& p, int b, int kvh, float qscale) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const uint4 u = *reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint8_t*>(p.q + head_row<G, MT>(p, b, kvh, h) * kD) +
            dim_off(v));
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          qf[h][4 * v + j] = mk2(bf16lo(wd[j]) * qscale, bf16hi(wd[j]) * qscale);
      }
  }
  // The same from the rotated query, q_rot [G][kD] fp32 in shared memory.
  __device__ __forceinline__ void load_q_rot(const float* q_rot, float qscale) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const float* src = q_rot + h * kD + dim_off(v) / 2;
        const float4 a = *reinterpret_cast<const float4*>(src);
        const float4 c = *reinterpret_cast<const float4*>(src + 4);
        qf[h][4 * v + 0] = mk2(a.x * qscale, a.y * qscale);
        qf[h][4 * v + 1] = mk2(a.z * qscale, a.w * qscale);
        qf[h][4 * v + 2] = mk2(c.x * qscale, c.y * qscale);
        qf[h][4 * v + 3] = mk2(c.z * qscale, c.w * qscale);
      }
  }
  __device__ __forceinline__ void reset() {
    m_run = -INFINITY;
    l_run = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int j = 0; j < NP; ++j) o[h][j] = mk2(0.f, 0.f);
  }
  // Scores (log2 domain) of this warp's keys of a tile; keys >= rows
  // are invalid (the rest of the stage may hold anything) and get -inf.
  // rows: keys of the tile this lane's head may see (all valid rows, or fewer
  // for an early token of a multi-token step)
  __device__ __forceinline__ void qk(const uint8_t* Ks, int rows, int warp, float (&sc)[IT]) {
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int key = warp * KPW + it * KPS + grp;
      f2 a[G];
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const uint4 kv = *reinterpret_cast<const uint4*>(Ks + key * kRowBytes + dim_off(v));
        f2 kf[4];
        unpack8x2(kv, kf);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            a[h] = (v == 0 && j == 0) ? mul2(qf[h][0], kf[0]) : fma2(qf[h][4 * v + j], kf[j], a[h]);
      }
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float lo, hi;
        brk2(a[h], lo, hi);
        acc[h] = lo + hi;
      }
      const float sv = reduce_key<G, LPK>(acc, lk);
      sc[it] = (key < rows) ? sv : -INFINITY;
    }
  }
  // Online softmax for head hd over the tile's scores -> probabilities pr.
  __device__ __forceinline__ void softmax(const float (&sc)[IT], float (&pr)[IT]) {
    float mx = sc[0];
#pragma unroll
    for (int it = 1; it < IT; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // Raise the running max only when it grows by more than 2^kTau (the
    // first valid tile always does): p may then reach 2^kTau, harmless in
    // fp32, and most tiles skip the rescale of o.
    const bool grow = mx > m_run + kTau;
    if (__any_sync(0xffffffffu, grow)) {
      const float alpha = grow ? ex2(m_run - mx) : 1.f;  // m_run = -inf: 0
      if (grow) m_run = mx;
      l_run *= alpha;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float ah = __shfl_sync(0xffffffffu, alpha, h << (LL - LG));
        const f2 a2 = mk2(ah, ah);
#pragma unroll
        for (int j = 0; j < NP; ++j) o[h][j] = mul2(o[h][j], a2);
      }
    }
    const float m_use = (m_run == -INFINITY) ? 0.f : m_run;  // no valid key yet
    float ps = 0.f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      pr[it] = ex2(sc[it] - m_use);
      ps += pr[it];
    }
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l_run += ps;
  }
  // o += p * v over this warp's keys of a tile.
  __device__ __forceinline__ void pv(const uint8_t* Vs, int rows, int warp, const float (&pr)[IT]) {
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int key = warp * KPW + it * KPS + grp;
      float ph[G];
#pragma unroll
      for (int h = 0; h < G; ++h)
        ph[h] = __shfl_sync(0xffffffffu, pr[it], (grp << LL) | (h << (LL - LG)));
      const bool valid = key < rows;  // invalid: p = 0, and v forced to 0 (stale smem)
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        uint4 vv = *reinterpret_cast<const uint4*>(Vs + key * kRowBytes + dim_off(v));
        vv.x = valid ? vv.x : 0u;
        vv.y = valid ? vv.y : 0u;
        vv.z = valid ? vv.z : 0u;
        vv.w = valid ? vv.w : 0u;
        f2 vf[4];
        unpack8x2(vv, vf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const f2 p2 = mk2(ph[h], ph[h]);
#pragma unroll
          for (int j = 0; j < 4; ++j) o[h][4 * v + j] = fma2(p2, vf[j], o[h][4 * v + j]);
        }
      }
    }
  }
  // One tile: scores, online softmax, P.V.
  __device__ __forceinline__ void tile(const uint8_t* Ks, const uint8_t* Vs, int rows, int rows_h,
                                       int warp) {
    float sc[IT], pr[IT];
    qk(Ks, rows_h, warp, sc);
    softmax(sc, pr);
    pv(Vs, rows, warp, pr);
  }
  // This warp's (m, l, o) -> merge buffers [warp][G][...]: the key groups
  // hold partial o for the same (m, l), so they are added first.
  __device__ __forceinline__ void stash(float* merge_o, float* merge_ml, int warp) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float lo, hi;
        brk2(o[h][j], lo, hi);
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
          lo += __shfl_xor_sync(0xffffffffu, lo, off);
          hi += __shfl_xor_sync(0xffffffffu, hi, off);
        }
        o[h][j] = mk2(lo, hi);
      }
    if (grp == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          float f[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) brk2(o[h][4 * v + j], f[2 * j], f[2 * j + 1]);
          float4* dst = reinterpret_cast<float4*>(
              reinterpret_cast<uint8_t*>(merge_o + (warp * G + h) * kD) + dim_off(v) * 2);
          dst[0] = make_float4(f[0], f[1], f[2], f[3]);
          dst[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
      if (lk == (hd << (LL - LG))) {
        merge_ml[(warp * G + hd) * 2 + 0] = m_run;
        merge_ml[(warp * G + hd) * 2 + 1] = l_run;
      }
    }
  }
};

// Merge the NW warps' partials of (head h, dim d): returns max M, sum Ls and
// unnormalised Os, all relative to M.
template <int NW, int G>
__device__ __forceinline__ void merge_warps(const float* merge_o, const float* merge_ml, int h,
                                            int d, float& M, float& Ls, float& Os) {
  M = -INFINITY;
#pragma unroll
  for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, merge_ml[(ww * G + h) * 2]);
  Ls = 0.f;
  Os = 0.f;
  const float Mu = (M == -INFINITY) ? 0.f : M;
#pragma unroll
  for (int ww = 0; ww < NW; ++ww) {
    const float e = ex2(merge_ml[(ww * G + h) * 2] - Mu);
    Ls = fmaf(merge_ml[(ww * G + h) * 2 + 1], e, Ls);
    Os = fmaf(merge_o[(ww * G + h) * kD + d], e, Os);
  }
}

// Producer (one thread): one tile's bulk copies.  With the fused append the
// segment's last tile ends with row pos = n-1, taken from k_new/v_new instead
// of the cache; a consumer warp rotates it if asked and writes it to the
// cache (fresh_row).  No other CTA reads that row.
__device__ __forceinline__ void produce_tile(const Params& p, uint8_t* stages, uint64_t* bars,
                                             int s, int b, int kvh, int k, int ntiles, int n,
                                             int lo) {
  // failure-path tests only: tile test_skip of the first segment is never
  // issued, so the bounded waits for it run out (ATTN_DEV_TIMEOUT)
  if (p.test_skip >= 0 && b == 0 && kvh == 0 && k == p.test_skip) return;
  const int rows = min(kTile, n - k * kTile);
  const size_t row0 = ((size_t)b * p.Hkv + kvh) * (size_t)p.L + (size_t)lo + (size_t)k * kTile;
  const bool fresh = p.k_new != nullptr && k == ntiles - 1;
  const int cache_rows = fresh ? rows - 1 : rows;
  const uint32_t full = smem_u32(&bars[s]);
  const uint32_t sK = smem_u32(stages + (size_t)s * 2 * kTileBytes);
  const uint32_t sV = sK + kTileBytes;
  mbar_arrive_expect_tx(full, 2u * (uint32_t)rows * kRowBytes);
  if (cache_rows > 0) {
    const uint32_t bytes = (uint32_t)cache_rows * kRowBytes;
    bulk_g2s(sK, p.k_cache + row0 * kRowBytes, bytes, full);
    bulk_g2s(sV, p.v_cache + row0 * kRowBytes, bytes, full);
  }
  if (fresh) {
    const size_t src = ((size_t)b * p.Hkv + kvh) * kRowBytes;
    const uint32_t off = (uint32_t)cache_rows * kRowBytes;
    bulk_g2s(sK + off, p.k_new + src, kRowBytes, full);
    bulk_g2s(sV + off, p.v_new + src, kRowBytes, full);
  }
}

// Rotary embedding of one segment, by the consumers.  rope_segment (all NC
// consumer threads, at the start of a segment, followed by a consumer
// barrier): the G query rows of the segment, rotated, into q_rot [G][kD] fp32,
// and the sequence's cos/sin row into rope_cs [2][kD].  rope_fresh_key (one
// warp, once the segment's last tile has landed): the appended key row of
// the tile rotated in place, lane l taking dims 4l..4l+3 and reading its
// partner dims 64 away before any lane writes.
template <int G, int NC>
__device__ __forceinline__ void rope_segment(const uint16_t* qb, const float* rc, const float* rs,
                                             float* q_rot, float* rope_cs, int ct) {
  constexpr int kH = kD / 2;
  for (int i = ct; i < G * kH; i += NC) {
    const int h = i / kH, d = i % kH;
    const uint16_t* qh = qb + (size_t)h * kD;
    const float x0 = __uint_as_float((uint32_t)qh[d] << 16);
    const float x1 = __uint_as_float((uint32_t)qh[d + kH] << 16);
    q_rot[h * kD + d] = rope1(x0, x1, rc[d], rs[d], true);
    q_rot[h * kD + d + kH] = rope1(x1, x0, rc[d + kH], rs[d + kH], false);
  }
  for (int i = ct; i < 2 * kD; i += NC) rope_cs[i] = i < kD ? rc[i] : rs[i - kD];
}

__device__ __forceinline__ void rope_fresh_key(uint8_t* row, const float* rope_cs, int lane) {
  const int d0 = 4 * lane;
  const uint2 a = *reinterpret_cast<const uint2*>(row + d0 * 2);
  const uint2 y2 = *reinterpret_cast<const uint2*>(row + (d0 ^ 64) * 2);
  __syncwarp();
  const float4 c4 = *reinterpret_cast<const float4*>(rope_cs + d0);
  const float4 s4 = *reinterpret_cast<const float4*>(rope_cs + kD + d0);
  float x[4] = {bf16lo(a.x), bf16hi(a.x), bf16lo(a.y), bf16hi(a.y)};
  const float y[4] = {bf16lo(y2.x), bf16hi(y2.x), bf16lo(y2.y), bf16hi(y2.y)};
  const float c[4] = {c4.x, c4.y, c4.z, c4.w};
  const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = rope1(x[j], y[j], c[j], sn[j], d0 < kD / 2);
  *reinterpret_cast<uint2*>(row + d0 * 2) =
      make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
}

// A consumer warp's wait for a tile, with the outcome made warp-uniform (the
// tile math uses full-warp shuffles, so either every lane goes on or every
// lane leaves the loop).
__device__ __forceinline__ bool consumer_wait(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t* status,
                                              int lane) {
  if (__all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag))) return true;
  if (lane == 0) {
    *abort_flag = 1;
    set_status(status, ATTN_DEV_TIMEOUT);
  }
  return false;
}

// The fused append's cache write: once a segment's last tile has landed, the
// appended K and V rows (its last row, rotated key included) go from shared
// memory to cache row pos = n-1, one 16-byte store per lane of one warp
// (lanes 0-15 the K row, 16-31 the V row).
__device__ __forceinline__ void write_fresh_rows(const Params& p, const uint8_t* Ks, int rows,
                                                 int b, int kvh, int pos, int lane) {
  const int c = lane & 15;
  const bool is_v = lane >= 16;
  const uint8_t* src = Ks + (is_v ? kTileBytes : 0) + (size_t)(rows - 1) * kRowBytes + c * 16;
  uint8_t* dst = (is_v ? p.v_cache : p.k_cache) +
                 (((size_t)b * p.Hkv + kvh) * (size_t)p.L + (size_t)pos) * kRowBytes + c * 16;
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}

// The appended row of a segment's last tile, by the one consumer warp whose
// keys include it (row rows-1): rotated in place first with the rotary
// embedding, then written to the cache.  No other warp reads the K row.
template <bool R>
__device__ __forceinline__ void fresh_row(const Params& p, uint8_t* Ks, int rows, int b, int kvh,
                                          int pos, const float* rope_cs, int lane) {
  if (R) {
    rope_fresh_key(Ks + (size_t)(rows - 1) * kRowBytes, rope_cs, lane);
    __syncwarp();
  }
  write_fresh_rows(p, Ks, rows, b, kvh, pos, lane);
}

// The rotation row of sequence b at position pos: row b of a [B, D] table,
// or row pos of an [L, D] table; null in kernels built without the rotary
// embedding (the compiler then drops the rotation code).
template <bool R>
__device__ __forceinline__ const float* rope_row(const Params& p, const float* t, int b, int pos) {
  return R ? t + (size_t)(p.rope_by_pos ? pos : b) * kD : nullptr;
}

// The position advance of a streaming step (p.advance non-null): called by
// warp 0 of every CTA once no thread of the CTA reads positions any more.
// The last CTA to arrive adds 1 to every position and rearms the ticket; its
// acquire orders those writes after every other CTA's reads.
__device__ __forceinline__ void advance_ticket(const Params& p, int lane) {
  uint32_t last = 0;
  if (lane == 0) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.ticket) : "memory");
    last = (old == gridDim.x - 1) ? 1u : 0u;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  if (!last) return;
  for (int b = lane; b < p.B; b += 32) p.advance[b] += 1;
  if (lane == 0) *p.ticket = 0u;
}

// NaN into every output row of sequence b (its S tokens' rows in
// multi-token decode).
__device__ __forceinline__ void write_nan_rows(const Params& p, int b, int S) {
  const uint4 nan4 = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
  uint4* o4 = reinterpret_cast<uint4*>(p.out + (size_t)b * S * p.Hq * kD);
  for (int i = 0; i < S * p.Hq * kD / 8; ++i) o4[i] = nan4;
}

__device__ __forceinline__ void store_bf16(uint16_t* dst, float v) {
  __nv_bfloat16 r = __float2bfloat16_rn(v);
  *dst = *reinterpret_cast<uint16_t*>(&r);
}

template <int G>
size_t smem_bytes(int B) {
  constexpr int NW = Cfg<G>::NW;
  return (size_t)kStages * 2 * kTileBytes + (2 * kStages + 2) * sizeof(uint64_t) +
         kMiscInts * sizeof(int) + (size_t)NW * G * 2 * sizeof(float) +
         (size_t)NW * G * kD * sizeof(float) + (2 + G) * kD * sizeof(float) +
         (size_t)(B + 1) * sizeof(int);
}

// ---------------------------------------------------------- stream-K mode --
template <int G, int M>
__global__ void __maxnreg__(Cfg<G>::kMaxRegs) decode_splitkv_kernel(const Params p) {
  constexpr bool R = (M & kModeRope) != 0, A = (M & kModeAdvance) != 0;
  constexpr bool MT = (M & kModeMulti) != 0;
  constexpr int NW = Cfg<G>::NW;
  constexpr int KPW = Cfg<G>::kKeysPerWarp;
  constexpr int NC = Cfg<G>::kConsumers;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * 2 * kTileBytes);
  int* misc = reinterpret_cast<int*>(bars + 2 * kStages + 2);  // after full, empty, csync, done
  float* merge_ml = reinterpret_cast<float*>(misc + kMiscInts);  // [NW][G][2]
  float* merge_o = merge_ml + NW * G * 2;                         // [NW][G][kD]
  float* rope_cs = merge_o + NW * G * kD;                         // [2][kD] cos, sin
  float* q_rot = rope_cs + 2 * kD;                                 // [G][kD]
  int* prefix = reinterpret_cast<int*>(q_rot + G * kD);            // [B+1]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, L = p.L;
  const int win = (M & kModeWindow) ? p.window : 0;
  const int shift = MT ? p.S - 1 : 0;  // positions[b] + shift: the last new token's row
  volatile int* abort_flag = misc;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);             // full: issuing thread's arrival + bytes
      mbar_init(smem_u32(&bars[kStages + s]), NW);  // empty: per consumer warp
    }
    mbar_init(smem_u32(&bars[2 * kStages]), NW);    // consumer barrier
    mbar_init(smem_u32(&bars[2 * kStages + 1]), NW + 1);  // done with positions
    misc[0] = 0;
    misc[1] = 0;
    fence_mbar_init();
  }
  // Launched with programmatic stream serialisation: everything above may run
  // while the previous kernel on the stream finishes; nothing written by it
  // (cache rows, positions, workspace counters) is read before this wait.
  grid_dependency_wait();
  grid_dependents_launch();

  // ---- tiles per sequence and their exclusive prefix sum (every CTA) ------
  int carry = 0;
  for (int base = 0; base < B; base += NC) {
    const int b = base + tid;
    int v = 0;
    if (tid < NC && b < B) {
      const int pos = p.positions[b] + shift;
      if (pos - shift >= 0 && pos < L) {
        int lo, n;
        attended_rows(pos, win, lo, n);
        v = (n - 1) / kTile + 1;  // ceil(n / kTile)
      } else if (b % gridDim.x == blockIdx.x) {
        // out-of-range position: flag it and make the sequence's output NaN
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
    if (lane == 31 && warp < NW) misc[8 + warp] = x;
    __syncthreads();
    int before = 0, chunk = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int s = misc[8 + w];
      before += (w < warp) ? s : 0;
      chunk += s;
    }
    if (tid < NC && b < B) prefix[b] = carry + before + x - v;
    carry += chunk;
    __syncthreads();
  }
  if (tid == 0) prefix[B] = carry;
  __syncthreads();

  const long long T = (long long)Hkv * carry;  // total tiles
  // Working CTAs: all of the grid, except when segments are short (on
  // average <= kWholeTiles tiles): then one CTA per segment, because a split
  // segment costs a partial round trip through L2, more than a few tiles.
  // Never more than T, so every working CTA gets >= 1 tile and the CTAs
  // covering a segment are exactly cta_of(first)..cta_of(last).
  const long long nseg = (long long)B * Hkv;
  long long gw = min((long long)gridDim.x, T);
  if (T <= (long long)kWholeTiles * nseg) gw = min(gw, nseg);
  const int Gd = (int)gw;
  if ((int)blockIdx.x >= Gd) {  // every thread is here, past its reads of positions
    if (A && warp == 0) advance_ticket(p, lane);
    return;
  }
  const long long t0 = T * blockIdx.x / Gd;
  const long long t1 = T * (blockIdx.x + 1) / Gd;

  // -------------------------------------------------------------- producer --
  if (warp == NW) {
    if (lane == 0) {
      Walk w;
      walk_init(w, t0, prefix, p.positions, B, Hkv, win, shift);
      long long i = 0;
      for (long long t = t0; t < t1; ++t, ++i) {
        const int s = (int)(i % kStages);
        const uint32_t u = (uint32_t)(i / kStages);
        if (i >= kStages &&
            !mbar_wait(smem_u32(&bars[kStages + s]), (u & 1u) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          set_status(p.status, ATTN_DEV_TIMEOUT);
          break;
        }
        produce_tile(p, stages, bars, s, w.b, w.kvh, w.k, w.ntiles, w.n, w.lo);
        walk_next(w, prefix, p.positions, B, Hkv, win, shift);
      }
      if (A) mbar_arrive(smem_u32(&bars[2 * kStages + 1]));  // no more reads of positions
    }
    return;
  }

  // ------------------------------------------------------------ consumers --
  Consumer<G> cs;
  cs.init(lane);
  ConsumerSync csync{smem_u32(&bars[2 * kStages]), abort_flag, p.status, 0u};
  Walk w;
  walk_init(w, t0, prefix, p.positions, B, Hkv, win, shift);
  const uint16_t* qb = p.q + ((size_t)w.b * p.Hq + (size_t)w.kvh * G) * kD;
  if (MT) cs.head_last = w.lo + w.n - 1 - shift + cs.hd / (G / p.S);
  if (R) {
    rope_segment<G, NC>(qb, rope_row<R>(p, p.rope_cos, w.b, w.lo + w.n - 1),
                        rope_row<R>(p, p.rope_sin, w.b, w.lo + w.n - 1), q_rot,
                        rope_cs, tid);
    consumer_bar<NC>();  // before any tile wait: every consumer warp gets here
    cs.load_q_rot(q_rot, p.qscale);
  } else {
    cs.template load_q<MT>(p, w.b, w.kvh, p.qscale);
  }
  cs.reset();

  long long i = 0;
  for (long long t = t0; t < t1; ++t, ++i) {
    const int s = (int)(i % kStages);
    const uint32_t u = (uint32_t)(i / kStages);
    if (!consumer_wait(smem_u32(&bars[s]), u & 1u, abort_flag, p.status, lane)) break;
    const int rows = min(kTile, w.n - w.k * kTile);
    uint8_t* Ks = stages + (size_t)s * 2 * kTileBytes;
    if (p.k_new != nullptr && w.k == w.ntiles - 1 && warp == (rows - 1) / KPW)
      fresh_row<R>(p, Ks, rows, w.b, w.kvh, w.lo + w.n - 1, rope_cs, lane);
    cs.tile(Ks, Ks + kTileBytes, rows,
            MT ? min(rows, cs.head_last + 1 - (w.lo + w.k * kTile)) : rows, warp);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[kStages + s]));  // the stage may be refilled
    const bool seg_end = (w.k == w.ntiles - 1) || (t == t1 - 1);

    // ---- end of this CTA's part of the segment: merge and emit ------------
    if (seg_end) {
      const int seg = w.b * Hkv + w.kvh;
      const long long seg_t0 = (long long)Hkv * prefix[w.b] + (long long)w.kvh * w.ntiles;
      const long long seg_t1 = seg_t0 + w.ntiles;
      const bool whole = seg_t0 >= t0 && seg_t1 <= t1;
      const int ct = tid;
      cs.stash(merge_o, merge_ml, warp);
      csync(lane);

      const int slot = blockIdx.x + seg;
      const int ob = w.b, okvh = w.kvh;  // the segment whose output this is
      for (int idx = ct; idx < G * kD; idx += NC) {
        const int h = idx / kD, d = idx % kD;
        float Mx, Ls, Os;
        merge_warps<NW, G>(merge_o, merge_ml, h, d, Mx, Ls, Os);
        if (whole) {
          store_bf16(p.out + head_row<G, MT>(p, ob, okvh, h) * kD + d, Os / Ls);
        } else {
          p.part_o[((size_t)slot * G + h) * kD + d] = Os;
          if (d == 0) {
            p.part_ml[((size_t)slot * G + h) * 2 + 0] = Mx;
            p.part_ml[((size_t)slot * G + h) * 2 + 1] = Ls;
          }
        }
      }
      if (!whole) {
        const int c_first = cta_of(seg_t0, T, Gd);
        const int c_last = cta_of(seg_t1 - 1, T, Gd);
        csync(lane);
        if (ct == 0) {
          // release: this CTA's partial (ordered before by the barrier) is
          // visible to whoever acquires the counter; acquire: the last
          // arrival sees every other CTA's partial
          unsigned old;
          asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                       : "=r"(old)
                       : "l"(&p.counters[seg])
                       : "memory");
          misc[1] = (old == (unsigned)(c_last - c_first)) ? 1 : 0;
        }
        csync(lane);
        if (misc[1]) {
          // last to arrive: merge the segment's partials.  Batches of 8
          // independent loads keep several L2 round trips in flight.
          for (int idx = ct; idx < G * kD; idx += NC) {
            const int h = idx / kD, d = idx % kD;
            float Mm = -INFINITY, Ls = 0.f, Os = 0.f;
            for (int c0 = c_first; c0 <= c_last; c0 += 8) {
              float mm[8], ll[8], oo[8];
#pragma unroll
              for (int uu = 0; uu < 8; ++uu) {
                const int c = c0 + uu;
                if (c <= c_last) {
                  const size_t sl = (size_t)(c + seg) * G + h;
                  mm[uu] = __ldcg(&p.part_ml[sl * 2]);
                  ll[uu] = __ldcg(&p.part_ml[sl * 2 + 1]);
                  oo[uu] = __ldcg(&p.part_o[sl * kD + d]);
                } else {
                  mm[uu] = -INFINITY;
                  ll[uu] = 0.f;
                  oo[uu] = 0.f;
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
                Os = fmaf(oo[uu], e, Os);
              }
              Mm = Mb;
            }
            store_bf16(p.out + head_row<G, MT>(p, ob, okvh, h) * kD + d, Os / Ls);
          }
          if (ct == 0) p.counters[seg] = 0u;  // ready for the next launch
        }
      }
      csync(lane);  // merge buffers are free again
      cs.reset();
    }
    walk_next(w, prefix, p.positions, B, Hkv, win, shift);
    if (w.k == 0 && t + 1 < t1) {
      // a new segment; every consumer has read q_rot and rope_cs of the last
      // one (seg_end's barriers came after), so they may be overwritten
      const uint16_t* qn = p.q + ((size_t)w.b * p.Hq + (size_t)w.kvh * G) * kD;
      if (R) {
        rope_segment<G, NC>(qn, rope_row<R>(p, p.rope_cos, w.b, w.lo + w.n - 1),
                            rope_row<R>(p, p.rope_sin, w.b, w.lo + w.n - 1),
                            q_rot, rope_cs, tid);
        csync(lane);
        cs.load_q_rot(q_rot, p.qscale);
      } else {
        cs.template load_q<MT>(p, w.b, w.kvh, p.qscale);
      }
      if (MT) cs.head_last = w.lo + w.n - 1 - shift + cs.hd / (G / p.S);
    }
  }

  if (*abort_flag) {
    // give copies that may still be in flight time to land before exit
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
  }
  if (A) {
    // this warp is done with positions; warp 0 waits for the producer and the
    // other consumers, then takes the CTA's ticket
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[2 * kStages + 1]));
    if (warp == 0) {
      mbar_wait(smem_u32(&bars[2 * kStages + 1]), 0u, abort_flag);
      advance_ticket(p, lane);
    }
  }
}

// ------------------------------------------------------------ cluster mode --
template <int G>
size_t cluster_smem_bytes() {
  constexpr int NW = Cfg<G>::NW;
  return (size_t)kStages * 2 * kTileBytes + (2 * kStages + 2) * sizeof(uint64_t) +
         kMiscInts * sizeof(int) + (size_t)NW * G * 2 * sizeof(float) +
         (size_t)NW * G * kD * sizeof(float) + (2 + G) * kD * sizeof(float) +
         (size_t)Cfg<G>::kMaxC * G * (kD + 2) * sizeof(float);
}

// Grid = B*Hkv clusters of C CTAs; cluster s handles segment s (sequence
// s / Hkv, KV head s % Hkv).
template <int G, int M>
__global__ void __maxnreg__(Cfg<G>::kMaxRegs) decode_cluster_kernel(const Params p) {
  constexpr bool R = (M & kModeRope) != 0, A = (M & kModeAdvance) != 0;
  constexpr bool MT = (M & kModeMulti) != 0;
  constexpr int NW = Cfg<G>::NW;
  constexpr int KPW = Cfg<G>::kKeysPerWarp;
  constexpr int NC = Cfg<G>::kConsumers;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * 2 * kTileBytes);
  int* misc = reinterpret_cast<int*>(bars + 2 * kStages + 2);  // after full, empty, csync, done
  float* merge_ml = reinterpret_cast<float*>(misc + kMiscInts);  // [NW][G][2]
  float* merge_o = merge_ml + NW * G * 2;                         // [NW][G][kD]
  float* rope_cs = merge_o + NW * G * kD;                         // [2][kD] cos, sin
  float* q_rot = rope_cs + 2 * kD;                                 // [G][kD]
  float* land_o = q_rot + G * kD;                    // [kMaxC][G][kD]: rank r's partial o
  float* land_ml = land_o + Cfg<G>::kMaxC * G * kD;  // [kMaxC][G][2]: its (max, sum)

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int seg = blockIdx.x / C;
  const int b = seg / p.Hkv, kvh = seg % p.Hkv;
  const int win = (M & kModeWindow) ? p.window : 0;
  const int shift = MT ? p.S - 1 : 0;  // positions[b] + shift: the last new token's row
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = misc;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[kStages + s]), NW);
    }
    mbar_init(smem_u32(&bars[2 * kStages]), NW);
    misc[0] = 0;
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_dependents_launch();
  const int pos = p.positions[b] + shift;
  if (pos - shift < 0 || pos >= p.L) {
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
  attended_rows(pos, win, lo, n);
  const int ntiles = (n - 1) / kTile + 1;
  const int k0 = (int)((long long)rank * ntiles / C);
  const int k1 = (int)((long long)(rank + 1) * ntiles / C);
  __syncthreads();  // barriers initialised
  // this CTA runs: the matching wait comes before any write into rank 0's
  // shared memory, so rank 0 is known to have started by then
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  if (warp == NW) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0;
        const int s = i % kStages;
        const uint32_t u = (uint32_t)(i / kStages);
        if (i >= kStages && !mbar_wait(smem_u32(&bars[kStages + s]), (u & 1u) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          set_status(p.status, ATTN_DEV_TIMEOUT);
          break;
        }
        produce_tile(p, stages, bars, s, b, kvh, k, ntiles, n, lo);
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers --
    Consumer<G> cs;
    cs.init(lane);
    ConsumerSync csync{smem_u32(&bars[2 * kStages]), abort_flag, p.status, 0u};
    const uint16_t* qb = p.q + ((size_t)b * p.Hq + (size_t)kvh * G) * kD;
    if (R) {
      rope_segment<G, NC>(qb, rope_row<R>(p, p.rope_cos, b, pos),
                          rope_row<R>(p, p.rope_sin, b, pos), q_rot,
                          rope_cs, tid);
      consumer_bar<NC>();  // before any tile wait: every consumer warp gets here
      cs.load_q_rot(q_rot, p.qscale);
    } else {
      cs.template load_q<MT>(p, b, kvh, p.qscale);
    }
    if (MT) cs.head_last = pos - shift + cs.hd / (G / p.S);
    cs.reset();
    for (int k = k0; k < k1; ++k) {
      const int i = k - k0;
      const int s = i % kStages;
      if (!consumer_wait(smem_u32(&bars[s]), (uint32_t)(i / kStages) & 1u, abort_flag, p.status,
                         lane))
        break;
      const int rows = min(kTile, n - k * kTile);
      uint8_t* Ks = stages + (size_t)s * 2 * kTileBytes;
      if (p.k_new != nullptr && k == ntiles - 1 && warp == (rows - 1) / KPW)
        fresh_row<R>(p, Ks, rows, b, kvh, pos, rope_cs, lane);
      cs.tile(Ks, Ks + kTileBytes, rows,
              MT ? min(rows, cs.head_last + 1 - (lo + k * kTile)) : rows, warp);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[kStages + s]));  // the stage may be refilled
    }
    // this CTA's warps' partials (max, sum, unnormalised o) merged below;
    // no tiles: (-inf, 0, 0)
    cs.stash(merge_o, merge_ml, warp);
    csync(lane);
  }

  // The CTA's partial goes straight into slot `rank` of rank 0's shared
  // memory (remote stores; nobody waits for them but the barrier below), so
  // rank 0 then merges from local memory and no CTA reads another's.
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (tid < NC) {
    float* to_o = cluster.map_shared_rank(land_o, 0) + rank * G * kD;
    float* to_ml = cluster.map_shared_rank(land_ml, 0) + rank * G * 2;
    for (int idx = tid; idx < G * kD; idx += NC) {
      const int h = idx / kD, d = idx % kD;
      float Mx, Ls, Os;
      merge_warps<NW, G>(merge_o, merge_ml, h, d, Mx, Ls, Os);
      to_o[h * kD + d] = Os;
      if (d == 0) {
        to_ml[h * 2 + 0] = Mx;
        to_ml[h * 2 + 1] = Ls;
      }
    }
  }

  cluster.sync();  // every rank's partial is in rank 0's shared memory
  if (rank == 0) {
    // weights 2^(m_r - M) / L per (rank, head): warp h reduces over the
    // ranks, lane r holding rank r's (max, sum); merge_ml is free by now
    float* wr = merge_ml;  // [C][G]
    if (warp < G) {
      const int h = warp;
      const bool in = lane < C;
      const float m = in ? land_ml[(lane * G + h) * 2] : -INFINITY;
      const float l = in ? land_ml[(lane * G + h) * 2 + 1] : 0.f;
      float Mx = m;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
      const float e = in ? ex2(m - Mx) : 0.f;  // a rank without tiles: 2^-inf = 0
      float Ls = l * e;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
      if (in) wr[lane * G + h] = e / Ls;
    }
    __syncthreads();
    for (int idx = tid; idx < G * kD; idx += blockDim.x) {
      const int h = idx / kD, d = idx % kD;
      float Os = 0.f;
#pragma unroll 4
      for (int r = 0; r < C; ++r) Os = fmaf(land_o[(r * G + h) * kD + d], wr[r * G + h], Os);
      store_bf16(p.out + head_row<G, MT>(p, b, kvh, h) * kD + d, Os);
    }
  }
  // no second cluster barrier: no CTA reads another's shared memory any more

  if (*abort_flag) {
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
  }
  // every thread read positions only before the cluster barrier above
  if (A && warp == 0) advance_ticket(p, lane);
}

// ------------------------------------------------------------------ host --


struct DevInfo {
  int num_sms = 0;
  bool configured[9] = {};               // per g
  int clusters[9][kMaxCluster + 1] = {};  // [g][C]: co-resident clusters of C CTAs
};
DevInfo g_dev[64];

DevInfo& dev_info(int* dev_out) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  *dev_out = dev;
  DevInfo& d = g_dev[dev];
  if (d.num_sms == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    d.num_sms = n;
  }
  return d;
}

template <int G>
int max_clusters(int C) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C * 64);
  cfg.blockDim = dim3(Cfg<G>::kThreads);
  cfg.dynamicSmemBytes = cluster_smem_bytes<G>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_cluster_kernel<G, 0>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int G, int M>
cudaError_t set_attributes(bool* big) {
  cudaError_t e = cudaFuncSetAttribute(decode_splitkv_kernel<G, M>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes<G>(kMaxB));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_cluster_kernel<G, M>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)cluster_smem_bytes<G>());
  if (e != cudaSuccess) return e;
  *big = cudaFuncSetAttribute(decode_cluster_kernel<G, M>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (!*big) cudaGetLastError();
  return cudaSuccess;
}

template <int G>
cudaError_t configure(DevInfo& d) {
  if (d.configured[G]) return cudaSuccess;
  bool big[6] = {};
  cudaError_t e = set_attributes<G, 0>(&big[0]);
  if (e == cudaSuccess) e = set_attributes<G, kModeRope>(&big[1]);
  if (e == cudaSuccess) e = set_attributes<G, kModeAdvance>(&big[2]);
  if (e == cudaSuccess) e = set_attributes<G, kModeRope | kModeAdvance>(&big[3]);
  if (e == cudaSuccess) e = set_attributes<G, kModeWindow>(&big[4]);
  if (e == cudaSuccess) e = set_attributes<G, kModeMulti>(&big[5]);
  if (e != cudaSuccess) return e;
  const bool big_all = big[0] && big[1] && big[2] && big[3] && big[4] && big[5];
  // How many clusters of each size can run at once (a cluster stays within
  // one GPC, so this is set by the SMs per GPC, not by the SM count).  All
  // variants have the same block, shared memory and register cap, so the
  // plain one stands for all.
  for (int c = 2; c <= kMaxCluster; ++c)
    d.clusters[G][c] = (c <= 8 || big_all) ? max_clusters<G>(c) : 0;
  d.configured[G] = true;
  return cudaSuccess;
}

// Cluster size for this launch: the largest in 8..kMaxC that lets every
// segment have its own co-resident cluster, or 0 (stream-K).
template <int G>
cudaError_t cluster_size(const Params& p, int* C) {
  int dev = 0;
  DevInfo& d = dev_info(&dev);
  cudaError_t e = configure<G>(d);
  if (e != cudaSuccess) return e;
  const long long nseg = (long long)p.B * p.Hkv;
  *C = 0;
  for (int c = Cfg<G>::kMaxC; c >= 8 && *C == 0; --c)
    if (nseg <= d.clusters[G][c]) *C = c;
  return cudaSuccess;
}

template <int G, int M>
cudaError_t launch_g(const Params& p, cudaStream_t stream) {
  int dev = 0;
  DevInfo& d = dev_info(&dev);
  int C = 0;
  cudaError_t e = cluster_size<G>(p, &C);
  if (e != cudaSuccess) return e;
  const long long nseg = (long long)p.B * p.Hkv;
  if (C > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nseg * C));
    cfg.blockDim = dim3(Cfg<G>::kThreads);
    cfg.dynamicSmemBytes = cluster_smem_bytes<G>();
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
    e = cudaLaunchKernelEx(&cfg, decode_cluster_kernel<G, M>, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  return launch_pdl(decode_splitkv_kernel<G, M>, dim3(min(kMaxGrid, d.num_sms)),
                    dim3(Cfg<G>::kThreads), smem_bytes<G>(p.B), stream, p);
}

// The variant for this launch.  The entry points use six combinations:
// plain, rotation, advance, rotation + advance, and the local window and the
// multi-token step alone.
template <int G>
cudaError_t launch_group(const Params& p, cudaStream_t stream) {
  const int mode = (p.rope_cos != nullptr ? kModeRope : 0) |
                   (p.advance != nullptr ? kModeAdvance : 0) | (p.window > 0 ? kModeWindow : 0) |
                   (p.S > 1 ? kModeMulti : 0);
  switch (mode) {
    case 0: return launch_g<G, 0>(p, stream);
    case kModeRope: return launch_g<G, kModeRope>(p, stream);
    case kModeAdvance: return launch_g<G, kModeAdvance>(p, stream);
    case kModeRope | kModeAdvance: return launch_g<G, kModeRope | kModeAdvance>(p, stream);
    case kModeWindow: return launch_g<G, kModeWindow>(p, stream);
    case kModeMulti: return launch_g<G, kModeMulti>(p, stream);
  }
  return cudaErrorInvalidValue;  // a combination no entry point makes
}

}  // namespace
}  // namespace gqa
