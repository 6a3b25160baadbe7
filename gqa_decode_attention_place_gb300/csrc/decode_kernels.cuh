// decode_kernels.cuh -- split-KV decode attention over a static KV cache with
// GQA, for group sizes g = 1, 2, 4 and 8 (8 without the rotary embedding):
// the kernels and their launch, included by one translation unit per group
// size (decode_g1.cu ... decode_g8.cu).  g = 16, and g = 8 with the rotary
// embedding, run on the tcgen05 tensor cores (decode_tc.cuh, which also uses
// the segment walk, helpers and tensor maps defined here).
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
//    cut into 128-row tiles, streamed by tiled TMA copies (two 64-dim boxes
//    per operand, 128-byte swizzle) into a 2-stage shared-memory ring
//    guarded by mbarriers (128 KB in flight per SM), issued by one producer
//    thread.  Each tile is read from HBM once and serves all g query heads
//    of its KV head.
//  * 8 consumer warps each take 16 keys of a tile and do both products with
//    warp-level tensor-core MMAs (mma.sync m16n8k16, bf16 in, fp32 out):
//    S = K q^T with the 16 keys as rows and the g heads as columns, then
//    O^T += V^T P^T with 16 dims per MMA.  The swizzle makes every
//    shared-memory read of both products conflict-free; P is moved from the
//    score layout to the operand layout by an 8x8 transpose in registers
//    (movmatrix) and enters as two bf16 parts (high and remainder), so the
//    product keeps about 16 bits of P.  The softmax is kept online in fp32
//    (running max and sum per head, base 2, scale*log2(e) applied to the fp32
//    scores).  On CUDA cores (fp32 FMAs, 16 lanes per key, shuffle
//    reductions) the same work took about 28 warp instructions per key;
//    here it takes about 7.
//  * Two ways to split a segment over CTAs, both computed on the device from
//    `positions` (one launch serves any positions; graph-capturable):
//    - cluster mode (few segments, e.g. B=1): one thread-block cluster of C
//      CTAs (8..16; the largest size that lets every
//      segment's cluster be resident at once) per segment; CTA rank r takes
//      tiles r, r+C, r+2C, ...  Tile r is then rank r's first whatever the
//      position, so its copy (and the q loads) go out before the position
//      is read.  Each CTA stores its partial (max, sum, unnormalised o)
//      straight into rank 0's shared memory (distributed shared memory);
//      after one cluster barrier rank 0 merges them locally in one pass --
//      no global scratch, no atomics.
//    - stream-K mode (many segments): all tiles of all segments form one flat
//      list; CTA c of a persistent grid (one per SM) takes
//      [c*T/G, (c+1)*T/G), balanced to one tile however ragged the batch is.
//      A segment split over CTAs is merged by the CTA that arrives last at
//      the segment's arrival counter (fp32 partials in the workspace; no
//      spin-wait).  A merge warp does every merge, so the consumer warps
//      only ever wait for tiles.
#pragma once

#include <cfloat>
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "decode_params.h"
#include "tcgen05.cuh"

namespace gqa {
namespace {

namespace cg = cooperative_groups;

constexpr int kD = kDecodeD;
constexpr int kTile = 128;                         // keys per pipeline stage
constexpr int kStages = 2;                         // stream-K ring (cluster mode: Cfg)
constexpr int kMaxRing = 3;                        // deepest ring of either mode
constexpr int kRowBytes = kD * 2;
constexpr int kTileBytes = kTile * kRowBytes;      // 32 KB per operand
constexpr int kHalf = kTile * 128;                 // one 64-dim box of an operand (16 KB)
constexpr int kMaxB = kDecodeMaxB;
constexpr int kMaxGrid = kDecodeMaxGrid;
constexpr int kMiscInts = 32;                      // [0] abort, [8..8+NW) scan
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

// The consumers: NW warps of 16 keys each per tile.
template <int G> struct Cfg {
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "these decode kernels serve g <= 8");
  static constexpr int NW = kTile / 16;
  // largest cluster: rank 0 keeps a landing slot for every rank's partial
  // (G x (kD + 2) floats each); 16 slots of 8 heads would not fit beside the
  // ring
  static constexpr int kMaxC = G == 8 ? 12 : 16;
  // the rotated query takes two MMA columns per head: g <= 4 only
  static constexpr bool kRope = 2 * G <= 8;
  // cluster mode's K/V ring: 3 stages where they fit beside rank 0's landing
  // slots (g <= 2), else 2
  static constexpr int kClusterStages = G <= 2 ? 3 : 2;
  static constexpr int kThreads = (NW + 1) * 32;  // + the producer warp
  static constexpr int kSKThreads = kThreads + 32;  // stream-K: + the merge warp
  static constexpr int kConsumers = NW * 32;
  static constexpr int kKeysPerWarp = kTile / NW;  // 16
  // registers per thread that still let one CTA of kSKThreads fit the SM
  // (the register file is handed out as if the block were a multiple of
  // 128 threads)
  static constexpr int kRegsFit = 65536 / ((kSKThreads + 127) / 128 * 128);
  static constexpr int kMaxRegs = (kRegsFit > 255 ? 255 : kRegsFit) & ~7;
};

// Barrier among the NW consumer warps.  It sits on an
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

// ---- warp-level tensor-core products (mma.sync m16n8k16, bf16 -> fp32) ----
// Fragment layouts (lane = 4*g + t): A (16x16, row-major) holds
// {A[g][2t..2t+1], A[g+8][2t..2t+1], A[g][2t+8..2t+9], A[g+8][2t+8..2t+9]};
// B (16x8, column-major) holds {B[2t..2t+1][g], B[2t+8..2t+9][g]}; the
// accumulator holds {C[g][2t], C[g][2t+1], C[g+8][2t], C[g+8][2t+1]}.  Each
// 32-bit register carries two bf16, the lower index in the low half.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Transpose of an 8x8 matrix of 16-bit values held as one row pair per lane
// (lane 4r + c holds row r, columns 2c and 2c+1).
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Bytes of a and b picked by `sel` (prmt): 0x5410 gives {a.lo, b.lo},
// 0x7632 gives {a.hi, b.hi}.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t word(const uint4& u, int i) {
  return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w;
}
// Byte offset of row r, dims 8c..8c+7 within one 64-dim box of a tile, as the
// 128-byte swizzle of the tiled copy lays it out (16-byte chunk c of row r
// sits at chunk c ^ (r mod 8); the stage buffers are 1024-byte aligned).
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }
// Byte offset of dims 8q..8q+7 (q = 0..15) of row r of a K or V tile.
__device__ __forceinline__ int tile_chunk(int r, int q) { return (q >> 3) * kHalf + sw128(r, q & 7); }

// Key (0..7, plus 8 for rows 8..15) that MMA row m of a warp's 16 stands
// for.  A 16-byte shared load is served per quarter warp (lanes 8i..8i+7,
// rows g = 2i and 2i+1): the K reads of those two rows must fall on opposite
// halves of the swizzle, so their keys differ in bit 2 (key_of(2i+1) =
// key_of(2i) ^ 4); the V reads of keys key_of(2t) (and of key_of(2t+1)),
// t = 0..3, must cover the four pairs {2k, 2k+1} once each.
__device__ __forceinline__ int key_of(int m) { return ((m & 6) | (m >> 2)) ^ ((m & 1) << 2); }

// Per-warp consumer state and math: one KV head's g query heads, 16 keys
// (kw .. kw+15) of each tile.  Lane 4g+t.
//  * Scores: S = K q^T, an m16n8k16 per 16 dims: the 16 keys are the rows,
//    heads the 8 columns (column h < g is head h; with the rotary embedding
//    column g+h carries the low bf16 part of rotated head h).  The 16 dims of
//    MMA step 2j+s are dims 64*(j/2) + 8*((j%2)*4 + t) + 4s .. +4 in lane t,
//    the same for the key rows (A) and for q (B), so one 16-byte read per key
//    row and lane feeds two MMAs and the 8 rows of each read hit 8 different
//    swizzle chunks.  MMA row m is key kw + key_of(m) (rows m+8: + 8), an
//    order that keeps these reads free of bank conflicts.  Lane 4g+t ends
//    with the scores of keys kw+key_of(g) and kw+8+key_of(g) for heads 2t
//    and 2t+1.
//  * P^T (keys x heads) is that score layout transposed in 8x8 blocks.
//  * Output: O^T += V^T P^T, m-block mb (0..7) holding dims 8g+mb (row g)
//    and 64+8g+mb (row g+8): lane 4g+t reads 16 bytes of dims 8g.. and
//    64+8g.. of the keys of MMA rows 2t, 2t+1, 2t+8, 2t+9 and pairs the
//    keys with prmt.  It accumulates O^T for those dims and heads 2t, 2t+1.
template <int G>
struct Consumer {
  static constexpr float kTau = 8.0f;  // a stale running max may lag by 2^8
  uint32_t qb[4][4];   // q^T as B operand, [dim group j][register]
  float o[8][4];       // O^T accumulators per m-block
  float m_run[2], l_run[2];  // heads 2t, 2t+1; l_run sums this lane's keys only
  int g, t;
  int head_last[2];    // multi-token decode: last row heads 2t, 2t+1 may see
  float qs;            // scale * log2(e), applied to the fp32 scores

  __device__ __forceinline__ void init(int lane) {
    g = lane >> 2;
    t = lane & 3;
  }
  // the G query rows of KV head kvh of sequence b (head_row), bf16 as stored
  template <bool MT>
  __device__ __forceinline__ void load_q(const DecodeParams& p, int b, int kvh, float qscale) {
    qs = qscale;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (g < G)
        u = *reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint8_t*>(p.q + head_row<G, MT>(p, b, kvh, g) * kD) +
            (j >> 1) * 128 + (((j & 1) * 4 + t) << 4));
      qb[j][0] = u.x;
      qb[j][1] = u.y;
      qb[j][2] = u.z;
      qb[j][3] = u.w;
    }
  }
  // The rotated query, straight from the segment's G query rows and the
  // rotation row (rc, rs: cos and sin, fp32): lane 4g+t rotates the 32 dims
  // it feeds to the MMA, each with its partner 64 dims away (rotate-half
  // form, one rounding per operation).  Column h < G takes the bf16
  // rounding of rotated head h, column G+h the rounding of what is left.
  // All of a lane's loads are independent: one round trip, no barrier.
  __device__ __forceinline__ void load_q_rope(const uint16_t* qrows, const float* rc,
                                              const float* rs, float qscale) {
    qs = qscale;
    const bool on = g < 2 * G;
    const uint16_t* qh = qrows + (size_t)(g < G ? g : g - G) * kD;
    // every load first (the compiler would otherwise interleave them with
    // the arithmetic, one round trip per dim group), then the rotations
    uint4 xv[4], yv[4];
    float4 cv[4][2], sv[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int d0 = (j >> 1) * 64 + ((j & 1) * 4 + t) * 8;
      xv[j] = yv[j] = make_uint4(0u, 0u, 0u, 0u);
      cv[j][0] = cv[j][1] = sv[j][0] = sv[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (on) {
        xv[j] = *reinterpret_cast<const uint4*>(qh + d0);
        yv[j] = *reinterpret_cast<const uint4*>(qh + (d0 ^ 64));
        cv[j][0] = *reinterpret_cast<const float4*>(rc + d0);
        cv[j][1] = *reinterpret_cast<const float4*>(rc + d0 + 4);
        sv[j][0] = *reinterpret_cast<const float4*>(rs + d0);
        sv[j][1] = *reinterpret_cast<const float4*>(rs + d0 + 4);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int d0 = (j >> 1) * 64 + ((j & 1) * 4 + t) * 8;
      const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
      const uint32_t yw[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
      const float cc[8] = {cv[j][0].x, cv[j][0].y, cv[j][0].z, cv[j][0].w,
                           cv[j][1].x, cv[j][1].y, cv[j][1].z, cv[j][1].w};
      const float ss[8] = {sv[j][0].x, sv[j][0].y, sv[j][0].z, sv[j][0].w,
                           sv[j][1].x, sv[j][1].y, sv[j][1].z, sv[j][1].w};
      const bool first = d0 < kD / 2;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float lo = rope1(bf16lo(xw[r]), bf16lo(yw[r]), cc[2 * r], ss[2 * r], first);
        const float hi = rope1(bf16hi(xw[r]), bf16hi(yw[r]), cc[2 * r + 1], ss[2 * r + 1], first);
        const uint32_t w = pack_bf16x2(lo, hi);
        qb[j][r] = !on ? 0u : g < G ? w : pack_bf16x2(lo - bf16lo(w), hi - bf16hi(w));
      }
    }
  }
  // The same operand from q already rotated (fp32 rows [G][kD], one per
  // head, in shared memory): column h < G gets the bf16 rounding of head h,
  // column G+h the rounding of what is left.  Bit-identical to load_q_rope.
  __device__ __forceinline__ void load_q_rotated(const float* rot, float qscale) {
    qs = qscale;
    const bool on = g < 2 * G;
    const float* qh = rot + (size_t)(g < G ? g : g - G) * kD;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int d0 = (j >> 1) * 64 + ((j & 1) * 4 + t) * 8;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (on) {
        a = *reinterpret_cast<const float4*>(qh + d0);
        b = *reinterpret_cast<const float4*>(qh + d0 + 4);
      }
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float lo = v[2 * r], hi = v[2 * r + 1];
        const uint32_t w = pack_bf16x2(lo, hi);
        qb[j][r] = !on ? 0u : g < G ? w : pack_bf16x2(lo - bf16lo(w), hi - bf16hi(w));
      }
    }
  }
  // multi-token decode: head h (token h / (G/S)) sees rows up to base + token
  __device__ __forceinline__ void set_last(int base, int S) {
#pragma unroll
    for (int e = 0; e < 2; ++e) head_last[e] = base + (2 * t + e) / (G / S);
  }
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m_run[e] = -INFINITY;
      l_run[e] = 0.f;
    }
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[mb][c] = 0.f;
  }
  // One tile: rows valid rows from absolute row row0 (multi-token decode:
  // head 2t+e only up to head_last[e]).  Rows past `rows` may hold anything.
  template <bool MT, bool R>
  __device__ __forceinline__ void tile(const uint8_t* Ks, const uint8_t* Vs, int rows, int row0,
                                       int warp) {
    const int kw = warp * 16;
    if (kw >= rows) return;  // no valid key for this warp (warp-uniform)
    const int pg = key_of(g);
    float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = (j & 1) * 4 + t;
      const uint8_t* base = Ks + (j >> 1) * kHalf;
      const uint4 ka = lds128(base + sw128(kw + pg, c));
      const uint4 kb = lds128(base + sw128(kw + pg + 8, c));
      mma16816(s, ka.x, kb.x, ka.y, kb.y, qb[j][0], qb[j][1]);
      mma16816(s2, ka.z, kb.z, ka.w, kb.w, qb[j][2], qb[j][3]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] += s2[i];
    if (R) {  // add the low parts' column G+h onto head h
      if (G == 1) {
        s[0] += s[1];
        s[2] += s[3];
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], G / 2);
      }
    }
    float x[4];  // log2-domain scores; invalid keys -inf
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int key = kw + pg + (i >> 1) * 8;
      const int lim = MT ? min(rows, head_last[i & 1] + 1 - row0) : rows;
      x[i] = key < lim ? s[i] * qs : -INFINITY;
    }
    float mx[2];
    bool grow[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[e] = fmaxf(x[e], x[2 + e]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], off));
      // raise the running max only when it grows by more than 2^kTau (the
      // first valid tile always does); columns past the heads never do
      grow[e] = (2 * t + e < G) && mx[e] > m_run[e] + kTau;
    }
    if (__any_sync(0xffffffffu, grow[0] || grow[1])) {
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        alpha[e] = grow[e] ? ex2(m_run[e] - mx[e]) : 1.f;  // m_run = -inf: 0
        if (grow[e]) m_run[e] = mx[e];
        l_run[e] *= alpha[e];
      }
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        o[mb][0] *= alpha[0];
        o[mb][1] *= alpha[1];
        o[mb][2] *= alpha[0];
        o[mb][3] *= alpha[1];
      }
    }
    float pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float mu = m_run[i & 1] == -INFINITY ? 0.f : m_run[i & 1];  // no valid key yet
      pr[i] = ex2(x[i] - mu);
    }
    l_run[0] += pr[0] + pr[2];
    l_run[1] += pr[1] + pr[3];
    // P^T as B operands: bf16 high parts and the bf16 rounding of the rest
    const uint32_t h0 = pack_bf16x2(pr[0], pr[1]), h1 = pack_bf16x2(pr[2], pr[3]);
    const uint32_t l0 = pack_bf16x2(pr[0] - bf16lo(h0), pr[1] - bf16hi(h0));
    const uint32_t l1 = pack_bf16x2(pr[2] - bf16lo(h1), pr[3] - bf16hi(h1));
    const uint32_t bh0 = movm_trans(h0), bh1 = movm_trans(h1);
    const uint32_t bl0 = movm_trans(l0), bl1 = movm_trans(l1);
    // MMA keys 2t, 2t+1, 2t+8, 2t+9
    const int vr[4] = {kw + key_of(2 * t), kw + key_of(2 * t + 1), kw + 8 + key_of(2 * t),
                       kw + 8 + key_of(2 * t + 1)};
    uint4 v[4][2];  // those keys' dims 8g.. and 64+8g..
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int h = 0; h < 2; ++h) v[k][h] = lds128(Vs + h * kHalf + sw128(vr[k], g));
    if (kw + 16 > rows) {  // V rows past the valid ones may be NaN: 0 * NaN would spread
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (vr[k] >= rows) v[k][0] = v[k][1] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const uint32_t sel = (mb & 1) ? 0x7632u : 0x5410u;
      const int w = mb >> 1;
      const uint32_t a0 = prmt(word(v[0][0], w), word(v[1][0], w), sel);
      const uint32_t a1 = prmt(word(v[0][1], w), word(v[1][1], w), sel);
      const uint32_t a2 = prmt(word(v[2][0], w), word(v[3][0], w), sel);
      const uint32_t a3 = prmt(word(v[2][1], w), word(v[3][1], w), sel);
      mma16816(o[mb], a0, a1, a2, a3, bh0, bh1);
      mma16816(o[mb], a0, a1, a2, a3, bl0, bl1);
    }
  }
  // This warp's (m, l, o) -> merge buffers [warp][G][...]
  __device__ __forceinline__ void stash(float* merge_o, float* merge_ml, int warp) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], off);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * t + e;
      if (h < G) {
        float* dst = merge_o + (warp * G + h) * kD + 8 * g;
        reinterpret_cast<float4*>(dst)[0] = make_float4(o[0][e], o[1][e], o[2][e], o[3][e]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(o[4][e], o[5][e], o[6][e], o[7][e]);
        reinterpret_cast<float4*>(dst + 64)[0] =
            make_float4(o[0][2 + e], o[1][2 + e], o[2][2 + e], o[3][2 + e]);
        reinterpret_cast<float4*>(dst + 64)[1] =
            make_float4(o[4][2 + e], o[5][2 + e], o[6][2 + e], o[7][2 + e]);
        if (g == 0) {
          merge_ml[(warp * G + h) * 2 + 0] = m_run[e];
          merge_ml[(warp * G + h) * 2 + 1] = l_run[e];
        }
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

// Producer (one thread): tile k of a segment, rows lo + k*kTile .. +kTile of
// sequence b, KV head kvh, as four tiled copies (K and V, two 64-dim boxes
// each).  Rows past the cache's end arrive as zeros; rows past the attended
// ones are masked by the consumers.  The transaction count is the full box.
__device__ __forceinline__ void produce_tile(const CUtensorMap* tmk, const CUtensorMap* tmv,
                                             const Params& p, uint8_t* stages, uint64_t* bars,
                                             int s, int b, int kvh, int k, int lo) {
  // failure-path tests only: tile test_skip of the first segment is never
  // issued, so the bounded waits for it run out (ATTN_DEV_TIMEOUT)
  if (p.test_skip >= 0 && b == 0 && kvh == 0 && k == p.test_skip) return;
  const uint32_t full = smem_u32(&bars[s]);
  const uint32_t sK = smem_u32(stages + (size_t)s * 2 * kTileBytes);
  const uint32_t sV = sK + kTileBytes;
  const int row = lo + k * kTile, z = b * p.Hkv + kvh;
  if (!range_ok(s >= 0 && s < kMaxRing && z >= 0 && z < p.B * p.Hkv && row >= 0 && row < p.L,
                p.status))
    return;
  mbar_arrive_expect_tx(full, 2u * kTileBytes);
  tma_load_3d(sK, tmk, 0, row, z, full);
  tma_load_3d(sK + kHalf, tmk, 64, row, z, full);
  tma_load_3d(sV, tmv, 0, row, z, full);
  tma_load_3d(sV + kHalf, tmv, 64, row, z, full);
}

// The rotation of the fused append's new key: the warp that writes the new
// rows stages, at the segment's start, the cos and sin values each of its
// lanes 0-15 will use (dims 8l..8l+7), in that lane's own 16 floats of
// rope_cs [2][kD].  No other lane reads them, so no barrier is needed.
__device__ __forceinline__ void stage_fresh_rope(float* rope_cs, const float* rc, const float* rs,
                                                 int lane) {
  if (lane < 16) {
    float4* dst = reinterpret_cast<float4*>(rope_cs + 16 * lane);
    dst[0] = *reinterpret_cast<const float4*>(rc + 8 * lane);
    dst[1] = *reinterpret_cast<const float4*>(rc + 8 * lane + 4);
    dst[2] = *reinterpret_cast<const float4*>(rs + 8 * lane);
    dst[3] = *reinterpret_cast<const float4*>(rs + 8 * lane + 4);
  }
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

// The fused append.  Lane l of the one consumer warp whose keys include the
// segment's last row (row pos = n-1 of the last tile) holds 16 bytes of the
// new rows: lanes 0-15 dims 8l..8l+7 of k_new, lanes 16-31 those of v_new
// (load_fresh, issued when the segment starts).  Once the tile has landed
// (its copy brought the stale cache row), fresh_row rotates the key if asked
// (the partner dims, 64 away, are in lane l^8), writes the row into the
// tile's shared memory and to cache row pos.  No other warp reads that row
// and no other CTA reads it in this launch.
__device__ __forceinline__ uint4 load_fresh(const Params& p, int b, int kvh, int lane) {
  const uint8_t* src = (lane < 16 ? p.k_new : p.v_new) +
                       ((size_t)b * p.Hkv + kvh) * kRowBytes + (lane & 15) * 16;
  return *reinterpret_cast<const uint4*>(src);
}

template <bool R>
__device__ __forceinline__ void fresh_row(const Params& p, uint8_t* Ks, int rows, int b, int kvh,
                                         int pos, const float* rope_cs, uint4 u, int lane) {
  const int q = lane & 15;  // 16-byte chunk of the row: dims 8q..8q+7
  if (R) {
    uint4 y;
    y.x = __shfl_xor_sync(0xffffffffu, u.x, 8);
    y.y = __shfl_xor_sync(0xffffffffu, u.y, 8);
    y.z = __shfl_xor_sync(0xffffffffu, u.z, 8);
    y.w = __shfl_xor_sync(0xffffffffu, u.w, 8);
    if (lane < 16) {
      const int d0 = 8 * q;
      const uint32_t xs[4] = {u.x, u.y, u.z, u.w}, ys[4] = {y.x, y.y, y.z, y.w};
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d = d0 + 2 * i;
        const float* cs = rope_cs + 16 * q;  // this lane's staged cos (0-7) and sin (8-15)
        r[i] = pack_bf16x2(
            rope1(bf16lo(xs[i]), bf16lo(ys[i]), cs[2 * i], cs[8 + 2 * i], d < kD / 2),
            rope1(bf16hi(xs[i]), bf16hi(ys[i]), cs[2 * i + 1], cs[8 + 2 * i + 1], d < kD / 2));
      }
      u = make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
  const bool is_v = lane >= 16;
  if (!range_ok(rows >= 1 && rows <= kTile && pos >= 0 && pos < p.L && b >= 0 && b < p.B &&
                    kvh >= 0 && kvh < p.Hkv,
                p.status))
    return;
  *reinterpret_cast<uint4*>(Ks + (is_v ? kTileBytes : 0) + tile_chunk(rows - 1, q)) = u;
  *reinterpret_cast<uint4*>((is_v ? p.v_cache : p.k_cache) +
                            (((size_t)b * p.Hkv + kvh) * (size_t)p.L + (size_t)pos) * kRowBytes +
                            q * 16) = u;
  __syncwarp();
}

// The rotation row of sequence b at position pos: row b of a [B, D] table,
// or row pos of an [L, D] table; null in kernels built without the rotary
// embedding (the compiler then drops the rotation code).
template <bool R>
__device__ __forceinline__ const float* rope_row(const Params& p, const float* t, int b, int pos) {
  return R ? t + (size_t)(p.rope_by_pos ? pos : b) * kD : nullptr;
}

// 1-D bulk copy global -> shared (the TMA engine; both addresses 16-byte
// aligned, size a multiple of 16), completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared memory of the rotary embedding in cluster mode: the inputs staged
// by bulk copies (G query rows, the new key row, the cos row, the sin row),
// then q rotated to fp32 rows [G][kD], then the new key rotated to bf16.
template <int G>
struct RopeStage {
  static constexpr int kIn = (G + 1) * kRowBytes + 2 * kD * 4;
  static constexpr int kRotQ = kIn;
  static constexpr int kRotK = kRotQ + G * kD * 4;
  static constexpr int kBytes = kRotK + kRowBytes;
};

// Copy the rotation's inputs into shared memory (one thread; bulk copies on
// the TMA engine, like the tiles: plain loads issued beside a tile's copy
// were measured to hold that copy back by about 1400 cycles).
template <int G>
__device__ __forceinline__ void stage_rope_inputs(uint8_t* area, const Params& p, int b, int kvh,
                                                  const float* rc, const float* rs, uint32_t bar) {
  mbar_arrive_expect_tx(bar, RopeStage<G>::kIn);
  bulk_copy(area, p.q + ((size_t)b * p.Hq + (size_t)kvh * G) * kD, G * kRowBytes, bar);
  bulk_copy(area + G * kRowBytes, p.k_new + ((size_t)b * p.Hkv + kvh) * kRowBytes, kRowBytes, bar);
  bulk_copy(area + (G + 1) * kRowBytes, rc, kD * 4, bar);
  bulk_copy(area + (G + 1) * kRowBytes + kD * 4, rs, kD * 4, bar);
}

// The producer warp's share of the rotary embedding, from the staged inputs:
// the G query rows rotated to fp32 (for the consumers' MMA operands) and the
// new key row rotated and rounded to bf16 (for the CTA whose part ends the
// segment).  Lane l takes dims 8(l%16)..+7 of rows l/16, l/16 + 2, ... (row
// G is the key); the partner dims are 64 away.  The same rounding, one IEEE
// operation at a time, as every other rotation here.
template <int G>
__device__ __forceinline__ void rotate_rows(uint8_t* area, int lane) {
  const int d0 = 8 * (lane & 15);
  const bool first = d0 < kD / 2;
  const float* rc = reinterpret_cast<const float*>(area + (G + 1) * kRowBytes);
  const float* rs = rc + kD;
  float* rot = reinterpret_cast<float*>(area + RopeStage<G>::kRotQ);
  uint8_t* rotk = area + RopeStage<G>::kRotK;
  const float4 c0 = *reinterpret_cast<const float4*>(rc + d0);
  const float4 c1 = *reinterpret_cast<const float4*>(rc + d0 + 4);
  const float4 s0 = *reinterpret_cast<const float4*>(rs + d0);
  const float4 s1 = *reinterpret_cast<const float4*>(rs + d0 + 4);
  const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  for (int r = lane >> 4; r <= G; r += 2) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(area + r * kRowBytes);
    const uint4 xv = *reinterpret_cast<const uint4*>(src + d0);
    const uint4 yv = *reinterpret_cast<const uint4*>(src + (d0 ^ 64));
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ys[4] = {yv.x, yv.y, yv.z, yv.w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = rope1(bf16lo(xs[i]), bf16lo(ys[i]), cc[2 * i], ss[2 * i], first);
      v[2 * i + 1] = rope1(bf16hi(xs[i]), bf16hi(ys[i]), cc[2 * i + 1], ss[2 * i + 1], first);
    }
    if (r < G) {
      float4* dst = reinterpret_cast<float4*>(rot + r * kD + d0);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      *reinterpret_cast<uint4*>(rotk + 2 * d0) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
  }
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
  // unsigned add: a position at INT_MAX wraps to a negative (rejected) one
  for (int b = lane; b < p.B; b += 32)
    p.advance[b] = (int32_t)((uint32_t)p.advance[b] + 1u);
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

// Element d of output row `row` (a head_row), checked in debug builds.
__device__ __forceinline__ void store_out(const Params& p, size_t row, int d, float v) {
  if (range_ok(row < (size_t)p.B * p.S * p.Hq && d >= 0 && d < kD, p.status))
    store_bf16(p.out + row * kD + d, v);
}

// Elements d0..d0+3 (d0 a multiple of 4) of output row `row`, each times
// `scale`: one 8-byte store.
__device__ __forceinline__ void store_out4(const Params& p, size_t row, int d0, float4 v,
                                           float scale) {
  if (range_ok(row < (size_t)p.B * p.S * p.Hq && d0 >= 0 && d0 + 3 < kD, p.status))
    *reinterpret_cast<uint2*>(p.out + row * kD + d0) =
        make_uint2(pack_bf16x2(v.x * scale, v.y * scale), pack_bf16x2(v.z * scale, v.w * scale));
}

// Stream-K shared memory: the ring, barriers, two merge slots of the NW
// warps' partials ([NW][G][kD] o, then [NW][G][2] max and sum), each warp's
// staged rotation values (rotary variants), and the tile prefix sum.
template <int G>
struct SKLayout {
  static constexpr int NW = Cfg<G>::NW;
  static constexpr int kBars = 2 * kStages + 6;  // full, empty, done, spare, merge full[2], empty[2]
  static constexpr int kBarDone = 2 * kStages;
  static constexpr int kBarMFull = 2 * kStages + 2;
  static constexpr int kBarMEmpty = 2 * kStages + 4;
  static constexpr int kSlotFloats = NW * G * (kD + 2);
  static constexpr int kRopeFloats = Cfg<G>::kRope ? NW * 256 : 0;  // [NW][16 lanes][16]
};

template <int G>
size_t smem_bytes(int B) {
  using Ly = SKLayout<G>;
  return (size_t)kStages * 2 * kTileBytes + Ly::kBars * sizeof(uint64_t) +
         kMiscInts * sizeof(int) + 2 * (size_t)Ly::kSlotFloats * sizeof(float) +
         (size_t)Ly::kRopeFloats * sizeof(float) + (size_t)(B + 1) * sizeof(int);
}

// ---------------------------------------------------------- stream-K mode --
// Roles: warps 0..NW-1 consume tiles, warp NW issues the copies, warp NW+1
// merges.  At the end of its part of a segment each consumer warp stashes
// its (max, sum, o) into a merge slot and goes on with the next segment; the
// merge warp combines the NW warps' partials and writes the output row, or,
// for a segment split over CTAs, the CTA's partial and -- if this CTA is the
// last to arrive -- the merge of all parts.  The consumers never wait for a
// merge (two slots), so merges are off the path that streams the cache.
//
// Tile order within the CTA's range [t0, t1): if its last segment starts
// inside the range and goes on past t1, that part comes first, the rest in
// order after it.  The other CTA holding that segment starts with its own
// part of it too, so the merge of every split segment happens early, and the
// range ends on a whole segment.
template <int G, int M>
__global__ void __maxnreg__(Cfg<G>::kMaxRegs) decode_splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                   const __grid_constant__ CUtensorMap tm_v,
                                                                   const Params p) {
  constexpr bool R = (M & kModeRope) != 0, A = (M & kModeAdvance) != 0;
  constexpr bool MT = (M & kModeMulti) != 0;
  using Ly = SKLayout<G>;
  constexpr int NW = Cfg<G>::NW;
  constexpr int KPW = Cfg<G>::kKeysPerWarp;
  constexpr int NC = Cfg<G>::kConsumers;
  constexpr int kMergeWarp = NW + 1;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * 2 * kTileBytes);
  int* misc = reinterpret_cast<int*>(bars + Ly::kBars);                 // [0] abort [8..8+NW) scan
  float* mslot = reinterpret_cast<float*>(misc + kMiscInts);            // [2][kSlotFloats]
  float* rope_cs = mslot + 2 * Ly::kSlotFloats;                         // [NW][16][16]
  int* prefix = reinterpret_cast<int*>(rope_cs + Ly::kRopeFloats);      // [B+1]

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
    mbar_init(smem_u32(&bars[Ly::kBarDone]), NW + 2);  // done with positions
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars[Ly::kBarMFull + s]), NW);  // every consumer warp stashed
      mbar_init(smem_u32(&bars[Ly::kBarMEmpty + s]), 1);  // the merge warp has read the slot
    }
    misc[0] = 0;
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
      const int p0 = p.positions[b];
      if (rows_in_cache(p0, shift, L)) {
        int lo, n;
        attended_rows(p0 + shift, win, lo, n);
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
  const long long n_t = t1 - t0;
  // processing order: tiles [tA, t1) first, then [t0, tA) (vJ = t1 - tA)
  long long tA = t0;
  {
    Walk wl;
    walk_init(wl, t1 - 1, prefix, p.positions, B, Hkv, win, shift);
    const long long s0 = t1 - 1 - wl.k;  // first tile of the last segment
    if (s0 > t0 && s0 + wl.ntiles > t1) tA = s0;
  }
  const long long vJ = t1 - tA;
  auto step = [&](Walk& w, long long v_next) {  // the walk for order index v_next
    if (v_next == vJ) walk_init(w, t0, prefix, p.positions, B, Hkv, win, shift);
    else walk_next(w, prefix, p.positions, B, Hkv, win, shift);
  };

  // -------------------------------------------------------------- producer --
  if (warp == NW) {
    if (lane == 0) {
      Walk w;
      walk_init(w, tA, prefix, p.positions, B, Hkv, win, shift);
      for (long long i = 0; i < n_t; ++i) {
        const int s = (int)(i % kStages);
        const uint32_t u = (uint32_t)(i / kStages);
        if (i >= kStages &&
            !mbar_wait(smem_u32(&bars[kStages + s]), (u & 1u) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          set_status(p.status, ATTN_DEV_TIMEOUT);
          break;
        }
        produce_tile(&tm_k, &tm_v, p, stages, bars, s, w.b, w.kvh, w.k, w.lo);
        if (i + 1 < n_t) step(w, i + 1);
      }
      if (A) mbar_arrive(smem_u32(&bars[Ly::kBarDone]));  // no more reads of positions
    }
    return;
  }

  // ---------------------------------------------------------- merge warp --
  if (warp == kMergeWarp) {
    Walk w;
    walk_init(w, tA, prefix, p.positions, B, Hkv, win, shift);
    const int d0 = 4 * lane;  // this lane's 4 dims of every head
    uint32_t k = 0;           // segment parts merged
    for (long long v = 0; v < n_t; ++k) {
      const long long v_end = v < vJ ? vJ : n_t;
      const long long len = min((long long)(w.ntiles - w.k), v_end - v);
      const int seg = w.b * Hkv + w.kvh;
      const long long seg_t0 = (long long)Hkv * prefix[w.b] + (long long)w.kvh * w.ntiles;
      const long long seg_t1 = seg_t0 + w.ntiles;
      const bool whole = seg_t0 >= t0 && seg_t1 <= t1;
      const int ob = w.b, okvh = w.kvh;
      if (!consumer_wait(smem_u32(&bars[Ly::kBarMFull + (k & 1)]), (k >> 1) & 1u, abort_flag,
                         p.status, lane))
        break;
      const float* so = mslot + (k & 1) * Ly::kSlotFloats;
      const float* sml = so + NW * G * kD;
      // combine the NW warps' partials of each head: max M, sum l, o (dims d0..d0+3)
      float hm[G], hl[G];
      float4 ho[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float Mx = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) Mx = fmaxf(Mx, sml[(ww * G + h) * 2]);
        const float Mu = Mx == -INFINITY ? 0.f : Mx;
        float l = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) {
          const float e = ex2(sml[(ww * G + h) * 2] - Mu);
          l = fmaf(sml[(ww * G + h) * 2 + 1], e, l);
          const float4 x = *reinterpret_cast<const float4*>(so + (ww * G + h) * kD + d0);
          o.x = fmaf(x.x, e, o.x);
          o.y = fmaf(x.y, e, o.y);
          o.z = fmaf(x.z, e, o.z);
          o.w = fmaf(x.w, e, o.w);
        }
        hm[h] = Mx;
        hl[h] = l;
        ho[h] = o;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[Ly::kBarMEmpty + (k & 1)]));  // slot free
      if (whole) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          store_out4(p, head_row<G, MT>(p, ob, okvh, h), d0, ho[h], 1.f / hl[h]);
      } else {
        // this CTA's partial, then the arrival; the last CTA to arrive merges
        const int c_first = cta_of(seg_t0, T, Gd);
        const int c_last = cta_of(seg_t1 - 1, T, Gd);
        const int slot = blockIdx.x + seg;
        if (range_ok(slot < kMaxGrid + B * Hkv, p.status)) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            *reinterpret_cast<float4*>(&p.part_o[((size_t)slot * G + h) * kD + d0]) = ho[h];
            if (lane == 0)
              *reinterpret_cast<float2*>(&p.part_ml[((size_t)slot * G + h) * 2]) =
                  make_float2(hm[h], hl[h]);
          }
        }
        // release: the warp's partial stores (ordered before by the warp
        // barrier) are visible to whoever acquires the counter; acquire: the
        // last arrival sees every other CTA's partial
        __threadfence();
        __syncwarp();
        uint32_t last = 0;
        if (lane == 0) {
          unsigned old;
          asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                       : "=r"(old)
                       : "l"(&p.counters[seg])
                       : "memory");
          last = (old == (unsigned)(c_last - c_first)) ? 1u : 0u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
#pragma unroll 1
          for (int h = 0; h < G; ++h) {
            float Mm = -INFINITY, Ls = 0.f;
            float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
            // batches of 4 independent loads keep several L2 round trips in flight
            for (int c0 = c_first; c0 <= c_last; c0 += 4) {
              float2 ml[4];
              float4 oo[4];
#pragma unroll
              for (int uu = 0; uu < 4; ++uu) {
                const int c = c0 + uu;
                if (c <= c_last && range_ok(c + seg < kMaxGrid + B * Hkv, p.status)) {
                  const size_t sl = (size_t)(c + seg) * G + h;
                  ml[uu] = __ldcg(reinterpret_cast<const float2*>(&p.part_ml[sl * 2]));
                  oo[uu] = __ldcg(reinterpret_cast<const float4*>(&p.part_o[sl * kD + d0]));
                } else {
                  ml[uu] = make_float2(-INFINITY, 0.f);
                  oo[uu] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
              }
              float Mb = Mm;
#pragma unroll
              for (int uu = 0; uu < 4; ++uu) Mb = fmaxf(Mb, ml[uu].x);
              const float Mu = Mb == -INFINITY ? 0.f : Mb;
              const float sc0 = ex2(Mm - Mu);  // Mm = -inf on the first batch: 0
              Ls *= sc0;
              Os.x *= sc0;
              Os.y *= sc0;
              Os.z *= sc0;
              Os.w *= sc0;
#pragma unroll
              for (int uu = 0; uu < 4; ++uu) {
                const float e = ex2(ml[uu].x - Mu);
                Ls = fmaf(ml[uu].y, e, Ls);
                Os.x = fmaf(oo[uu].x, e, Os.x);
                Os.y = fmaf(oo[uu].y, e, Os.y);
                Os.z = fmaf(oo[uu].z, e, Os.z);
                Os.w = fmaf(oo[uu].w, e, Os.w);
              }
              Mm = Mb;
            }
            store_out4(p, head_row<G, MT>(p, ob, okvh, h), d0, Os, 1.f / Ls);
          }
          if (lane == 0) p.counters[seg] = 0u;  // ready for the next launch
        }
      }
      v += len;
      if (v < n_t) {
        if (v == vJ) {
          walk_init(w, t0, prefix, p.positions, B, Hkv, win, shift);
        } else {
          w.k = w.ntiles - 1;  // on to the next segment
          walk_next(w, prefix, p.positions, B, Hkv, win, shift);
        }
      }
    }
    if (A) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[Ly::kBarDone]));  // no more reads of positions
    }
    return;
  }

  // ------------------------------------------------------------ consumers --
  Consumer<G> cs;
  cs.init(lane);
  float* my_rope_cs = rope_cs + (R ? warp * 256 : 0);  // this warp's staged cos, sin
  Walk w;
  walk_init(w, tA, prefix, p.positions, B, Hkv, win, shift);
  const uint16_t* qb = p.q + ((size_t)w.b * p.Hq + (size_t)w.kvh * G) * kD;
  if (MT) cs.set_last(w.lo + w.n - 1 - shift, p.S);
  // fused append: this warp writes the segment's new rows if the segment's
  // last tile is in this CTA's range and its last row among the warp's keys
  // (a segment whose part comes first in the order ends past t1)
  auto owns_fresh = [&](const Walk& ww, long long t) {
    return p.k_new != nullptr && t + (ww.ntiles - 1 - ww.k) < t1 &&
           warp == (ww.n - 1 - (ww.ntiles - 1) * kTile) / KPW;
  };
  bool own_fresh = owns_fresh(w, tA);
  uint4 fk = own_fresh ? load_fresh(p, w.b, w.kvh, lane) : make_uint4(0u, 0u, 0u, 0u);
  if (R) {
    const float* rc = rope_row<R>(p, p.rope_cos, w.b, w.lo + w.n - 1);
    const float* rs = rope_row<R>(p, p.rope_sin, w.b, w.lo + w.n - 1);
    cs.load_q_rope(qb, rc, rs, p.qscale);
    if (own_fresh) stage_fresh_rope(my_rope_cs, rc, rs, lane);
  } else {
    cs.template load_q<MT>(p, w.b, w.kvh, p.qscale);
  }
  cs.reset();

  uint32_t kseg = 0;  // segment parts stashed
  for (long long i = 0; i < n_t; ++i) {
    const int s = (int)(i % kStages);
    const uint32_t u = (uint32_t)(i / kStages);
    if (!consumer_wait(smem_u32(&bars[s]), u & 1u, abort_flag, p.status, lane)) break;
    const int rows = min(kTile, w.n - w.k * kTile);
    uint8_t* Ks = stages + (size_t)s * 2 * kTileBytes;
    if (own_fresh && w.k == w.ntiles - 1)
      fresh_row<R>(p, Ks, rows, w.b, w.kvh, w.lo + w.n - 1, my_rope_cs, fk, lane);
    cs.template tile<MT, R>(Ks, Ks + kTileBytes, rows, w.lo + w.k * kTile, warp);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[kStages + s]));  // the stage may be refilled
    const bool more = i + 1 < n_t;
    const bool seg_end = (w.k == w.ntiles - 1) || i + 1 == vJ || !more;
    Walk wn = w;
    if (more) step(wn, i + 1);

    // ---- end of this CTA's part of the segment: hand it to the merge warp --
    if (seg_end) {
      if (more) {
        // the next segment's q (rotated if asked) and new rows only need
        // loads: they go out now and land while this part is stashed
        const long long tn = (i + 1) < vJ ? tA + i + 1 : t0 + (i + 1 - vJ);
        if (R)
          cs.load_q_rope(p.q + ((size_t)wn.b * p.Hq + (size_t)wn.kvh * G) * kD,
                         rope_row<R>(p, p.rope_cos, wn.b, wn.lo + wn.n - 1),
                         rope_row<R>(p, p.rope_sin, wn.b, wn.lo + wn.n - 1), p.qscale);
        else
          cs.template load_q<MT>(p, wn.b, wn.kvh, p.qscale);
        if (MT) cs.set_last(wn.lo + wn.n - 1 - shift, p.S);
        own_fresh = owns_fresh(wn, tn);
        if (own_fresh) {
          fk = load_fresh(p, wn.b, wn.kvh, lane);
          if (R)
            stage_fresh_rope(my_rope_cs, rope_row<R>(p, p.rope_cos, wn.b, wn.lo + wn.n - 1),
                             rope_row<R>(p, p.rope_sin, wn.b, wn.lo + wn.n - 1), lane);
        }
      }
      // the slot's previous segment has been read by the merge warp
      if (kseg >= 2 && !consumer_wait(smem_u32(&bars[Ly::kBarMEmpty + (kseg & 1)]),
                                      ((kseg >> 1) - 1) & 1u, abort_flag, p.status, lane))
        break;
      float* so = mslot + (kseg & 1) * Ly::kSlotFloats;
      cs.stash(so, so + NW * G * kD, warp);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[Ly::kBarMFull + (kseg & 1)]));
      ++kseg;
      cs.reset();
    }
    w = wn;
  }

  if (*abort_flag) {
    // give copies that may still be in flight time to land before exit
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
  }
  if (A) {
    // this warp is done with positions; warp 0 waits for the producer, the
    // merge warp and the other consumers, then takes the CTA's ticket
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[Ly::kBarDone]));
    if (warp == 0) {
      mbar_wait(smem_u32(&bars[Ly::kBarDone]), 0u, abort_flag);
      advance_ticket(p, lane);
    }
  }
}

// ------------------------------------------------------------ cluster mode --
template <int G>
size_t cluster_smem_bytes() {
  constexpr int NW = Cfg<G>::NW;
  constexpr int NS = Cfg<G>::kClusterStages;
  return (size_t)NS * 2 * kTileBytes + (2 * NS + 2) * sizeof(uint64_t) +
         kMiscInts * sizeof(int) + (size_t)NW * G * 2 * sizeof(float) +
         (size_t)NW * G * kD * sizeof(float) + 2 * kD * sizeof(float) +
         (size_t)Cfg<G>::kMaxC * G * (kD + 2) * sizeof(float) +
         (Cfg<G>::kRope ? (size_t)RopeStage<G>::kBytes : 0) + 2 * sizeof(uint64_t);
}

// Grid = B*Hkv clusters of C CTAs; cluster s handles segment s (sequence
// s / Hkv, KV head s % Hkv).
template <int G, int M>
__global__ void __maxnreg__(Cfg<G>::kMaxRegs)
    decode_cluster_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const Params p) {
  constexpr bool R = (M & kModeRope) != 0, A = (M & kModeAdvance) != 0;
  constexpr bool MT = (M & kModeMulti) != 0;
  constexpr int NW = Cfg<G>::NW;
  constexpr int NS = Cfg<G>::kClusterStages;  // ring stages in shared memory
  // stages the ring uses: with the rotary embedding two, so that its staging
  // copies meet a shorter TMA queue (a third stage measured slower there)
  constexpr int NR = R ? 2 : NS;
  constexpr int KPW = Cfg<G>::kKeysPerWarp;
  constexpr int NC = Cfg<G>::kConsumers;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * 2 * kTileBytes);
  int* misc = reinterpret_cast<int*>(bars + 2 * NS + 2);  // after full, empty, csync, done
  float* merge_ml = reinterpret_cast<float*>(misc + kMiscInts);  // [NW][G][2]
  float* merge_o = merge_ml + NW * G * 2;                         // [NW][G][kD]
  float* rope_cs = merge_o + NW * G * kD;                         // [2][kD] staged cos, sin
  float* land_o = rope_cs + 2 * kD;                  // [kMaxC][G][kD]: rank r's partial o
  float* land_ml = land_o + Cfg<G>::kMaxC * G * kD;  // [kMaxC][G][2]: its (max, sum)
  // rotation (RopeStage): staged inputs, q and the new key rotated, and two
  // mbarriers: the staging copies landed; the producer warp wrote the rotations
  uint8_t* q_stage = reinterpret_cast<uint8_t*>(land_ml + Cfg<G>::kMaxC * G * 2);
  const float* rot_q = reinterpret_cast<const float*>(q_stage + RopeStage<G>::kRotQ);
  const uint8_t* rot_k = q_stage + RopeStage<G>::kRotK;
  uint64_t* stage_bar = reinterpret_cast<uint64_t*>(
      q_stage + (Cfg<G>::kRope ? RopeStage<G>::kBytes : 0));
  uint64_t* q_stage_bar = stage_bar + 1;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int seg = blockIdx.x / C;
  const int b = seg / p.Hkv, kvh = seg % p.Hkv;
  const int win = (M & kModeWindow) ? p.window : 0;
  const int shift = MT ? p.S - 1 : 0;  // positions[b] + shift: the last new token's row
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool producer = tid == NW * 32;
  volatile int* abort_flag = misc;

  if (producer) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[NS + s]), NW);
    }
    mbar_init(smem_u32(&bars[2 * NS]), NW);
    mbar_init(smem_u32(stage_bar), 1);
    mbar_init(smem_u32(q_stage_bar), 1);
    misc[0] = 0;
    fence_mbar_init();
  }
  // The step's own small inputs (this segment's q rows, new rows and
  // position) are often cold in HBM: warm them into L2 while the previous
  // kernel finishes.  An L2 prefetch returns no data, and L2 is where every
  // write lands first, so anything the previous kernel still writes there
  // is what the loads after the wait see.
  if (warp == 0 && lane < 8) {
    const uint8_t* qrow = reinterpret_cast<const uint8_t*>(
        p.q + head_row<G, MT>(p, b, kvh, 0) * kD);
    if (!MT && lane < G * 2) prefetch_l2(qrow + lane * 128);  // G contiguous rows of 256 bytes
    if (p.k_new != nullptr && lane < 4) {
      const size_t off = ((size_t)b * p.Hkv + kvh) * kRowBytes + (lane & 1) * 128;
      prefetch_l2((lane < 2 ? p.k_new : p.v_new) + off);
    }
    if (lane == 7) prefetch_l2(p.positions + b);
  }
  if (R && warp == 1 && lane < 8 && !p.rope_by_pos)  // per-sequence rotation rows: 2 x 512 bytes
    prefetch_l2((lane < 4 ? p.rope_cos : p.rope_sin) + (size_t)b * kD + (lane & 3) * 32);
  grid_dependency_wait();
  grid_dependents_launch();
  // Rank r's first tile is tile r whatever the position (rows from 0 without
  // a local window), so its copy goes out before the position is read, and
  // so does q, loaded; with the rotary embedding and per-sequence rotation
  // rows the rotation's inputs are copied in just before it, and the producer
  // warp rotates q and the new key once it has issued the next tile.  If the
  // position leaves rank r without tiles, the copies only have to land
  // before the CTA exits.
  const bool early = !(M & kModeWindow) && rank * kTile < p.L;
  // the rotation's inputs (a few KB) go ahead of the tile, so that they land,
  // and are rotated, while the tile is still in flight
  if (R && !p.rope_by_pos && producer)  // rotation rows known before the position
    stage_rope_inputs<G>(q_stage, p, b, kvh, rope_row<R>(p, p.rope_cos, b, 0),
                         rope_row<R>(p, p.rope_sin, b, 0), smem_u32(stage_bar));
  if (early && producer) produce_tile(&tm_k, &tm_v, p, stages, bars, 0, b, kvh, rank, 0);
  // the position's load goes out first; its value is used after the q setup
  const int pos0 = p.positions[b];
  Consumer<G> cs;
  if (warp < NW) {
    cs.init(lane);
    if (!R) cs.template load_q<MT>(p, b, kvh, p.qscale);
  }
  if (!rows_in_cache(pos0, shift, p.L)) {
    // the same for every CTA of the cluster: all leave, no cluster barrier
    if (R && !p.rope_by_pos && producer) mbar_wait(smem_u32(stage_bar), 0u, abort_flag);
    if (early && producer) mbar_wait(smem_u32(&bars[0]), 0u, abort_flag);
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
  const int pos = pos0 + shift;
  int lo, n;
  attended_rows(pos, win, lo, n);
  const int ntiles = (n - 1) / kTile + 1;
  __syncthreads();  // barriers initialised
  // this CTA runs: the matching wait comes before any write into rank 0's
  // shared memory, so rank 0 is known to have started by then
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  if (warp == NW) {
    // ------------------------------------------------------------ producer --
    // the tiles of the first round (free stages, no wait), then the rotation,
    // then the rest
    if (lane == 0) {
      if (R && p.rope_by_pos)  // the rotation rows are the position's
        stage_rope_inputs<G>(q_stage, p, b, kvh, rope_row<R>(p, p.rope_cos, b, pos),
                             rope_row<R>(p, p.rope_sin, b, pos), smem_u32(stage_bar));
      int i = 0;
      for (int k = rank; k < ntiles && i < NR; k += C, ++i)
        if (i > 0 || !early) produce_tile(&tm_k, &tm_v, p, stages, bars, i, b, kvh, k, lo);
    }
    __syncwarp();
    if (R) {
      if (__all_sync(0xffffffffu, mbar_wait(smem_u32(stage_bar), 0u, abort_flag))) {
        rotate_rows<G>(q_stage, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(q_stage_bar));  // the consumers may read them
      } else if (lane == 0) {
        *abort_flag = 1;
        set_status(p.status, ATTN_DEV_TIMEOUT);
      }
    }
    if (lane == 0) {
      int i = NR;
      for (int k = rank + NR * C; k < ntiles; k += C, ++i) {
        const int s = i % NR;
        const uint32_t u = (uint32_t)(i / NR);
        if (!mbar_wait(smem_u32(&bars[NS + s]), (u & 1u) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          set_status(p.status, ATTN_DEV_TIMEOUT);
          break;
        }
        produce_tile(&tm_k, &tm_v, p, stages, bars, s, b, kvh, k, lo);
      }
      // a first copy that no consumer waits for lands before the CTA exits
      if (early && rank >= ntiles) mbar_wait(smem_u32(&bars[0]), 0u, abort_flag);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers --
    ConsumerSync csync{smem_u32(&bars[2 * NS]), abort_flag, p.status, 0u};
    if (MT) cs.set_last(pos - shift, p.S);
    // fused append: the warp whose keys include the last row of the last
    // tile, in the rank that takes that tile, writes the new rows
    const bool own_fresh = p.k_new != nullptr && (ntiles - 1) % C == rank &&
                           warp == (n - 1 - (ntiles - 1) * kTile) / KPW;
    const uint4 fk = own_fresh ? load_fresh(p, b, kvh, lane) : make_uint4(0u, 0u, 0u, 0u);
    cs.reset();
    int i = 0;
    for (int k = rank; k < ntiles; k += C, ++i) {
      const int s = i % NR;
      if (!consumer_wait(smem_u32(&bars[s]), (uint32_t)(i / NR) & 1u, abort_flag, p.status,
                         lane))
        break;
      if (R && i == 0) {  // the operand from the producer warp's rotated q
        if (!consumer_wait(smem_u32(q_stage_bar), 0u, abort_flag, p.status, lane)) break;
        cs.load_q_rotated(rot_q, p.qscale);
      }
      const int rows = min(kTile, n - k * kTile);
      uint8_t* Ks = stages + (size_t)s * 2 * kTileBytes;
      if (own_fresh && k == ntiles - 1)  // with the rotation: the key rotated by the producer
        fresh_row<false>(p, Ks, rows, b, kvh, pos, rope_cs,
                         (R && lane < 16) ? reinterpret_cast<const uint4*>(rot_k)[lane] : fk,
                         lane);
      cs.template tile<MT, R>(Ks, Ks + kTileBytes, rows, lo + k * kTile, warp);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[NS + s]));  // the stage may be refilled
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
  if (tid < NC && range_ok(rank < Cfg<G>::kMaxC && C <= Cfg<G>::kMaxC, p.status)) {
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
    // One pass per output element: the max over the ranks, then the C
    // weights 2^(m_r - M) (independent of one another, so they issue back to
    // back), the sum and the weighted partials.  A rank without tiles has
    // m = -inf and weighs 0; some rank always has a valid key.
    for (int idx = tid; idx < G * kD; idx += blockDim.x) {
      const int h = idx / kD, d = idx % kD;
      float m[Cfg<G>::kMaxC];
      float Mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < Cfg<G>::kMaxC; ++r) {
        m[r] = r < C ? land_ml[(r * G + h) * 2] : -INFINITY;
        Mx = fmaxf(Mx, m[r]);
      }
      float Ls = 0.f, Os = 0.f;
#pragma unroll
      for (int r = 0; r < Cfg<G>::kMaxC; ++r) {
        if (r < C) {
          const float e = ex2(m[r] - Mx);
          Ls = fmaf(land_ml[(r * G + h) * 2 + 1], e, Ls);
          Os = fmaf(land_o[(r * G + h) * kD + d], e, Os);
        }
      }
      store_out(p, head_row<G, MT>(p, b, kvh, h), d, Os / Ls);
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
  bool configured[9] = {};               // per g (1, 2, 4 and 8)
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
  if constexpr (Cfg<G>::kRope) {
    if (e == cudaSuccess) e = set_attributes<G, kModeRope>(&big[1]);
    if (e == cudaSuccess) e = set_attributes<G, kModeRope | kModeAdvance>(&big[3]);
  } else {
    big[1] = big[3] = true;
  }
  if (e == cudaSuccess) e = set_attributes<G, kModeAdvance>(&big[2]);
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
  const int force = g_decode_test_cluster;  // schedule tests only
  if (force >= 0) {
    // a cluster size these kernels cannot launch is refused, not replaced
    if (force > Cfg<G>::kMaxC || (force > 8 && d.clusters[G][force] == 0))
      return cudaErrorNotSupported;
    *C = force;
  }
  return cudaSuccess;
}

// A cache [B*Hkv, L, 128] bf16 as a 3-D tensor map (dims, rows, segments);
// box 64 dims x 128 rows x 1, 128-byte swizzle: one column block of a tile.
// Rows past L read as zeros.  The last few maps are kept per host thread.
bool cache_map(CUtensorMap* m, const void* ptr, int L, long long segs) {
  struct Entry {
    const void* ptr;
    int L;
    long long segs;
    CUtensorMap map;
  };
  static thread_local Entry cache[4] = {};
  static thread_local int next = 0;
  for (const Entry& e : cache)
    if (e.ptr == ptr && e.L == L && e.segs == segs) {
      *m = e.map;
      return true;
    }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)segs};
  cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)kRowBytes * (cuuint64_t)L};
  cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = Entry{ptr, L, segs, *m};
  next = (next + 1) % 4;
  return true;
}

template <int G, int M>
cudaError_t launch_g(const Params& p, cudaStream_t stream) {
  int dev = 0;
  DevInfo& d = dev_info(&dev);
  const long long nseg = (long long)p.B * p.Hkv;
  CUtensorMap mk, mv;
  if (!cache_map(&mk, p.k_cache, p.L, nseg) || !cache_map(&mv, p.v_cache, p.L, nseg))
    return cudaErrorInvalidValue;
  int C = 0;
  cudaError_t e = cluster_size<G>(p, &C);
  if (e != cudaSuccess) return e;
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
    e = cudaLaunchKernelEx(&cfg, decode_cluster_kernel<G, M>, mk, mv, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  return launch_pdl(decode_splitkv_kernel<G, M>, dim3(min(kMaxGrid, d.num_sms)),
                    dim3(Cfg<G>::kSKThreads), smem_bytes<G>(p.B), stream, mk, mv, p);
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
    case kModeAdvance: return launch_g<G, kModeAdvance>(p, stream);
    case kModeWindow: return launch_g<G, kModeWindow>(p, stream);
    case kModeMulti: return launch_g<G, kModeMulti>(p, stream);
  }
  if constexpr (Cfg<G>::kRope) {
    if (mode == kModeRope) return launch_g<G, kModeRope>(p, stream);
    if (mode == (kModeRope | kModeAdvance)) return launch_g<G, kModeRope | kModeAdvance>(p, stream);
  }
  return cudaErrorInvalidValue;  // a combination no entry point makes (or rotation at g = 8)
}

}  // namespace
}  // namespace gqa
