/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: in-place static-KV-cache GQA decode
 * attention and causal prefill over a cached prefix, for NVIDIA GB300
 * (sm_103a).
 *
 * Where the operations come from (page title, section):
 *   - "MiniCPM4 `forward_step` Attention Performance Fix", section 4.1: each
 *     decode step writes the new key/value row of every KV head in place into
 *     a preallocated static cache [B, Hkv, max_len, D] at position_id, then
 *     attends the query heads (GQA, enable_gqa) over cache rows
 *     0..position_id only -- no boolean mask and no full-length copy
 *     (section 3).  Sections 2.4 and 6.4: the per-step cost must grow with
 *     position_id + 1, not with max_len.
 *   - "step14_3 -- batched attention", sections "problem" and
 *     "F.scaled_dot_product_attention": prefill of S new tokens whose K/V
 *     include the cached prefix, token-major layout [tokens, heads, d_head].
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps device memory.
 *   - Tensors are bf16 (raw 16-bit storage, `const void*`), dense, row-major,
 *     with the shapes given per call.  Every tensor pointer must be 16-byte
 *     aligned.
 *   - GQA: query head h reads KV head h / g, g = Hq / Hkv (contiguous groups,
 *     the repeat-KV convention).
 *   - Kernels are launched with programmatic stream serialisation: a launch
 *     may start its prologue while the previous kernel on `stream` drains,
 *     and waits for that kernel's writes before reading any input.
 *   - Every call is asynchronous on `stream` and returns an int status
 *     (ATTN_OK or an ATTN_ERR_* code).  Argument errors are found on the host
 *     before anything is launched; nothing is then written.  ATTN_ERR_CUDA means
 *     a launch failed; attn_last_cuda_error() returns the CUDA error code.
 *   - Errors that only the device can see (a position outside [0, max_len))
 *     never trap: the affected sequence is skipped, decode writes NaN to its
 *     output rows, and a bit is set in the device status word kept in the
 *     decode workspace (read it with attn_read_device_status).
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define ATTN_OK                0
#define ATTN_ERR_INVALID_ARG   1  /* null pointer, non-positive size, Hq % Hkv != 0,
                                     pointer not 16-byte aligned, start_pos < 0 */
#define ATTN_ERR_UNSUPPORTED   2  /* a size the library has no kernel for (see each call) */
#define ATTN_ERR_WORKSPACE     3  /* workspace null or smaller than attn_decode_workspace_size() */
#define ATTN_ERR_CUDA          4  /* a CUDA runtime call or launch failed */
#define ATTN_ERR_DEVICE        5  /* attn_read_device_status: the device flagged a fault */

/* Bits of the device status word (attn_read_device_status(..., &bits)). */
#define ATTN_DEV_BAD_POSITION  0x1u  /* some positions[b] was outside [0, max_len) */
#define ATTN_DEV_TIMEOUT       0x2u  /* a pipeline wait gave up (the kernel returned early) */
#define ATTN_DEV_RANGE         0x4u  /* debug builds only (attn_debug_build() == 1): an
                                        index-derived access (a bulk-copy tile coordinate,
                                        a cluster landing slot, a partial-result slot, an
                                        output or new-row address) failed its range check
                                        and was skipped; the launch's outputs are undefined */

/*
 * attn_kv_append -- the in-place cache write of the decode page, section 4.1
 * (key_cache[:, :, position_id, :] = key_states; same for values), with one
 * position per sequence.
 *
 *   k_new, v_new : [B, Hkv, D] bf16, the new rows.
 *   positions    : [B] int32, device memory; row positions[b] of every KV head
 *                  of sequence b is overwritten.
 *   k_cache,
 *   v_cache      : [B, Hkv, L, D] bf16, modified in place.  Every other byte
 *                  is left untouched (bit-exact copy of the new rows).
 *   D            : multiple of 8 (16-byte rows), 8 <= D <= 256.
 *
 * A position outside [0, L) skips that sequence's write (no other effect;
 * attn_decode_step with the same positions reports it).
 */
int attn_kv_append(const void* k_new, const void* v_new, const int32_t* positions,
                   void* k_cache, void* v_cache,
                   int B, int Hkv, int L, int D, cudaStream_t stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode_step
 * needs for these sizes (split-KV partial results, per-(sequence, KV head)
 * arrival counters and the device status word).  Returns 0 if the sizes are
 * invalid or unsupported.  The workspace must be zero-filled before its first
 * use (e.g. cudaMemsetAsync).  Every call leaves its arrival counters at zero
 * again, so later calls with the same (B, Hq, Hkv, D) can reuse it as is; zero
 * it again before using it with other sizes, or after a call that reported
 * ATTN_DEV_TIMEOUT.  Calls that share a workspace must not overlap in time.
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int L, int D);

/*
 * attn_decode_step -- sliced decode attention of the decode page, sections 3
 * and 4.1: for every sequence b and query head h,
 *     out[b,h,:] = softmax_j(scale * q[b,h,:] . K[b,h/g,j,:]) V[b,h/g,j,:]
 * over j = 0..positions[b] inclusive.  Rows above positions[b] are never read
 * (they may hold anything, NaN included).  Call attn_kv_append first for the
 * step's new row (the page writes the row, then attends).
 *
 *   q         : [B, Hq, D] bf16 (one query token per sequence).
 *   positions : [B] int32, device memory.
 *   k_cache,
 *   v_cache   : [B, Hkv, L, D] bf16.
 *   scale     : fp32 score scale (the page's default is 1/sqrt(D)).
 *   out       : [B, Hq, D] bf16 (= [B, Hq*D]), fp32 softmax and accumulation,
 *               rounded to nearest even.  Both contractions of a tile run
 *               on tensor cores with bf16 operands and fp32 accumulation:
 *               per warp (mma.sync) for g <= 8, with the probabilities
 *               entering P.V as two bf16 parts (about 16 bits); on the
 *               tcgen05 tensor cores for g = 16 (and for the rotary entry
 *               points at g = 8), with the probabilities rounded to bf16
 *               before P.V.
 *   workspace : device buffer of at least attn_decode_workspace_size(...)
 *               bytes, zero-filled before first use (see above).
 *
 * Supported: D == 128; g = Hq / Hkv in {1, 2, 4, 8, 16} (g = 16 on the
 * tcgen05 tensor cores); 1 <= B <= 8192;
 * 1 <= L <= 2^24.  Work is split over the attended rows only, so the cost of
 * a step follows sum_b (positions[b] + 1), not B * L.
 */
int attn_decode_step(const void* q, const int32_t* positions,
                     const void* k_cache, const void* v_cache,
                     int B, int Hq, int Hkv, int L, int D, float scale,
                     void* out, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/*
 * attn_decode_step_append -- one decode step of the decode page, section 4.1,
 * in one launch: the cache write of attn_kv_append followed by the attention
 * of attn_decode_step.  Results are those of the two calls in that order:
 * row positions[b] of every KV head of sequence b becomes k_new/v_new
 * (bit-exact) and out is attention over rows 0..positions[b], the new row
 * included.  The new rows are fed to the attention straight from k_new/v_new
 * and written to the cache in the same launch.  For g <= 8 the new row goes
 * through the tile like any cache row, so out is bit-identical to the two
 * calls; on the tcgen05 kernels (g = 16) its score and value are folded in
 * fp32 beside the tile, so out agrees with the two calls to rounding.
 *
 *   q            : [B, Hq, D] bf16.
 *   k_new, v_new : [B, Hkv, D] bf16.
 *   positions    : [B] int32, device memory.
 *   k_cache,
 *   v_cache      : [B, Hkv, L, D] bf16, row positions[b] written in place.
 *   out, workspace, scale and supported sizes: as attn_decode_step.
 *
 * A position outside [0, L) writes nothing for that sequence, gives NaN
 * output rows and sets ATTN_DEV_BAD_POSITION.
 */
int attn_decode_step_append(const void* q, const void* k_new, const void* v_new,
                            const int32_t* positions, void* k_cache, void* v_cache,
                            int B, int Hq, int Hkv, int L, int D, float scale,
                            void* out, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * attn_decode_step_rope_append -- attn_decode_step_append with the rotary
 * position embedding applied first, as the decode page's forward_step does
 * (section 4.1: apply_rotary_pos_emb(q, k, cos, sin) runs before the cache
 * write).  The page does not define the rotation; this library takes the
 * rotate-half form, for every dim d of a row x:
 *     x'[d] = x[d]*cos[d] - x[d+D/2]*sin[d]          for d <  D/2
 *     x'[d] = x[d]*cos[d] + x[d-D/2]*sin[d]          for d >= D/2
 * in fp32, each product and the sum rounded separately (no fused
 * multiply-add).  The rotated key is rounded to bf16 (nearest even) and that
 * is what the cache row holds; the rotated query is kept in fp32 for the
 * attention.  v_new is appended unrotated.
 *
 *   cos, sin : [B, D] fp32, device memory, 16-byte aligned; row b is the
 *              rotation for sequence b at positions[b] (the caller computes
 *              it, so any frequency base or scaling works).  Read only.
 *   all other arguments, sizes and errors: as attn_decode_step_append.
 *
 * Errors: ATTN_ERR_INVALID_ARG also for a null or misaligned cos or sin;
 * ATTN_ERR_UNSUPPORTED for g = 16 (the rotation serves g <= 8: the
 * tensor-core kernels carry the rotated query as two bf16 rows per head).
 */
int attn_decode_step_rope_append(const void* q, const void* k_new, const void* v_new,
                                 const float* cos, const float* sin,
                                 const int32_t* positions, void* k_cache, void* v_cache,
                                 int B, int Hq, int Hkv, int L, int D, float scale,
                                 void* out, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * attn_decode_step_window -- decode attention over a local window: each
 * sequence attends only its last `window` cache rows up to its position,
 *     rows max(0, positions[b] - window + 1) .. positions[b] inclusive,
 * so the current token is always included.  The decode pages name the
 * variant without defining it; this reading takes the W most recent rows.
 * Rows outside the window are never read.  The cost of a step follows
 * min(window, positions[b] + 1), not the position.
 *
 *   k_new, v_new : [B, Hkv, D] bf16 rows to append at positions[b] first
 *                  (as attn_decode_step_append), or both null to attend only
 *                  (as attn_decode_step).
 *   window       : > 0; window >= positions[b] + 1 is the full decode.
 *   all other arguments, sizes and errors: as attn_decode_step_append.
 *
 * Errors: ATTN_ERR_INVALID_ARG also for window <= 0, or for exactly one of
 * k_new and v_new null.
 */
int attn_decode_step_window(const void* q, const void* k_new, const void* v_new,
                            const int32_t* positions, void* k_cache, void* v_cache,
                            int B, int Hq, int Hkv, int L, int D, int window, float scale,
                            void* out, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * attn_decode_multi -- multi-token decode: S new tokens per sequence (for
 * example draft tokens to verify) in one launch.  Token t of sequence b sits
 * at position positions[b] + t and attends cache rows
 * 0 .. positions[b] + t: the earlier new tokens and itself, not the later
 * ones.  Each KV byte is read once for all S tokens and g query heads of its
 * KV head.  This is the decode page's step for several tokens at once.  The
 * causal rule for the new block is the prefill page's, aligned to the
 * bottom-right corner.
 *
 *   q            : [B, S, Hq, D] bf16.
 *   k_new, v_new : [B, S, Hkv, D] bf16, appended first at rows
 *                  positions[b] .. positions[b] + S - 1 (a separate launch
 *                  ahead of the attention); or both null when the cache
 *                  already holds them.
 *   positions    : [B] int32, device memory: the first new token's position.
 *   out          : [B, S, Hq, D] bf16.
 *   workspace    : at least attn_decode_workspace_size(B, S * Hq, Hkv, L, D)
 *                  bytes, zero-filled before first use.
 *   Supported: D == 128; S * g in {1, 2, 4, 8, 16}; other limits as
 *   attn_decode_step.  S == 1 is attn_decode_step (after the append).
 *
 * A sequence whose positions[b] + S - 1 falls outside [0, L) gets NaN in all
 * of its output rows, no cache write, and ATTN_DEV_BAD_POSITION.
 * Errors: ATTN_ERR_INVALID_ARG for null or misaligned pointers, exactly one
 * of k_new and v_new null, or non-positive sizes; ATTN_ERR_UNSUPPORTED when
 * S * g is not 1, 2, 4, 8 or 16; ATTN_ERR_WORKSPACE as above.
 */
int attn_decode_multi(const void* q, const void* k_new, const void* v_new,
                      const int32_t* positions, void* k_cache, void* v_cache,
                      int B, int S, int Hq, int Hkv, int L, int D, float scale,
                      void* out, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/*
 * attn_decode_stream_step -- one step of a streaming decode loop that a CUDA
 * graph can capture once and replay unchanged.  It performs the fused step of
 * attn_decode_step_append (preceded by the rotary embedding of
 * attn_decode_step_rope_append when tables are given), then adds one to every
 * positions[b] on the device.  The decode page calls forward_step once per
 * new token at position_id, the next one at position_id + 1 (section 4.1);
 * keeping that counter on the device lets one captured launch serve every
 * step of the loop.
 *
 *   positions : [B] int32, device memory.  It is read as this step's positions,
 *               then every entry is incremented by one, out-of-range ones
 *               included.  The increment happens after every part of the
 *               launch has read them, so the result is the same as a step at
 *               the old positions followed by a host-side increment.
 *   cos_table,
 *   sin_table : [L, D] fp32, device memory, 16-byte aligned, or both null for
 *               no rotation.  Row p is the rotation at position p; the step
 *               uses row positions[b] for sequence b.  Read only.
 *   all other arguments, sizes and errors: as attn_decode_step_append.  The
 *   step uses a counter in the workspace and leaves it at zero again.
 *
 * Errors: ATTN_ERR_INVALID_ARG also when exactly one of cos_table and
 * sin_table is null, or either is misaligned; ATTN_ERR_UNSUPPORTED for the
 * rotation at g = 16 (as attn_decode_step_rope_append).
 */
int attn_decode_stream_step(const void* q, const void* k_new, const void* v_new,
                            const float* cos_table, const float* sin_table,
                            int32_t* positions, void* k_cache, void* v_cache,
                            int B, int Hq, int Hkv, int L, int D, float scale,
                            void* out, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * attn_decode_step_noalloc -- attn_decode_step without a workspace argument.
 * The decode page has no counterpart: this entry point exists for callers
 * that cannot call cudaMalloc, for example plugin or embedded hosts that own
 * all device memory and hand the library none, and real-time streaming loops
 * where the device-wide synchronisation an allocation can imply would stall
 * playback.  It allocates nothing: its split-KV scratch is a fixed 16 MiB
 * device array inside the library, which every GPU that loads the library
 * holds until the process exits.
 *
 * Arguments, supported sizes and results are those of attn_decode_step.
 * Sizes whose attn_decode_workspace_size() exceeds 16 MiB (16777216 bytes)
 * are rejected with ATTN_ERR_WORKSPACE (B=256, Hq=64, Hkv=8, D=128 needs about
 * 12.8 MB and fits).  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) while that device is current, and so does
 * the first call after the device's context was replaced (cudaDeviceReset).
 * The lookup is guarded by a mutex, so host threads may make their first
 * calls at the same time.  Every
 * call first clears the array's status word and arrival counters with
 * cudaMemsetAsync on `stream`.  All calls share the one array, so calls that
 * overlap on the GPU (other streams, other host threads) race and give wrong
 * results; serialise them.  The device status word is not readable for this
 * variant: an out-of-range position still gives NaN output rows.
 */
int attn_decode_step_noalloc(const void* q, const int32_t* positions,
                             const void* k_cache, const void* v_cache,
                             int B, int Hq, int Hkv, int L, int D, float scale,
                             void* out, cudaStream_t stream);

/*
 * attn_prefill_causal -- causal prefill over a cached prefix (prefill page,
 * section "F.scaled_dot_product_attention"; decode page section 5: batch
 * prefill is causal).  New token i (absolute position start_pos + i) attends
 * keys 0..start_pos + i: the causal mask aligned to the bottom-right corner.
 *
 *   q         : [S, Hq, d] bf16, the S new tokens (token-major).
 *   k, v      : [start_pos + S, Hkv, d] bf16, cached prefix rows first.
 *   out       : [S, Hq, d] bf16 (= [S, Hq*d]).
 *
 * Supported: d == 64 or d == 128; g = Hq / Hkv >= 1; S >= 0 (S == 0 does nothing);
 * start_pos >= 0; start_pos + S < 2^31.  QK^T and PV run on the tcgen05
 * tensor cores (bf16 operands, fp32 accumulation in tensor memory).
 *
 * Every wait in the kernel is bounded: one that runs out ends the launch
 * early, leaves some output rows unwritten, and is counted on the device;
 * attn_read_prefill_status reads (and clears) that count.
 */
int attn_prefill_causal(const void* q, const void* k, const void* v,
                        int S, int start_pos, int Hq, int Hkv, int d, float scale,
                        void* out, cudaStream_t stream);

/*
 * attn_read_prefill_status -- synchronise `stream`, read into *timeouts the
 * number of prefill waits that gave up since the last call on this device,
 * clear it, and return ATTN_OK if there were none, ATTN_ERR_DEVICE if there
 * were, or ATTN_ERR_CUDA.  `timeouts` may be NULL.
 */
int attn_read_prefill_status(uint32_t* timeouts, cudaStream_t stream);

/*
 * attn_read_device_status -- synchronise `stream`, read the device status
 * word from a decode workspace into *bits (ATTN_DEV_* flags), clear it, and
 * return ATTN_OK if no bit was set, ATTN_ERR_DEVICE if one was, or
 * ATTN_ERR_INVALID_ARG / ATTN_ERR_CUDA.  `bits` may be NULL.
 */
int attn_read_device_status(void* workspace, uint32_t* bits, cudaStream_t stream);

/* Human-readable name of a status code (static string; never NULL). */
const char* attn_status_string(int status);

/* CUDA error code (cudaError_t as int) of the last ATTN_ERR_CUDA on this host
 * thread, 0 if none. */
int attn_last_cuda_error(void);

/*
 * attn_test_skip_tile -- for tests of the failure path only.  From the next
 * decode launch on, the bulk copy of tile `tile` (128 rows) of the first
 * (sequence, KV head) segment is never issued.  The waits for that tile
 * therefore run out: every wait in the kernels gives up
 * after 500 ms.  The kernel then sets ATTN_DEV_TIMEOUT in the workspace's
 * status word and returns, and the CUDA context stays usable; the outputs of
 * that launch are undefined, and its workspace must be zero-filled again
 * before reuse.  -1 (the default) turns this off.  Process-wide and not
 * thread-safe.
 * Errors: ATTN_ERR_INVALID_ARG for tile < -1.
 */
int attn_test_skip_tile(int tile);

/*
 * attn_test_force_schedule -- for tests of the split schedules only.  From
 * the next decode launch on, every segment (sequence, KV head) is split the
 * way `cluster` says instead of by the automatic choice: 0 = stream-K (all
 * tiles of all segments in one flat list over a persistent grid, split
 * segments merged through the workspace), C in 1..16 = cluster mode with
 * clusters of C CTAs (one cluster per segment, partials merged in rank 0's
 * shared memory), -1 (the default) = automatic.  Results agree with the
 * automatic choice up to the rounding of a different merge order.  A decode
 * call whose kernel cannot run clusters of C (too many landing slots for its
 * shared memory, or more than 8 where the device allows no larger clusters)
 * fails with ATTN_ERR_CUDA (cudaErrorNotSupported).  Process-wide and not
 * thread-safe.
 * Errors: ATTN_ERR_INVALID_ARG for cluster < -1 or > 16.
 */
int attn_test_force_schedule(int cluster);

/*
 * attn_debug_build -- 1 if this library was compiled with the device range
 * checks (-DGQA_DEBUG), else 0.  In such a build every decode kernel checks
 * the index-derived addresses named under ATTN_DEV_RANGE before it uses them,
 * and both prefill kernels check their bulk-copy tile coordinates and output
 * rows; a failed check skips the access and records it (no trap, no assert).
 * Release builds contain no checks.
 */
int attn_debug_build(void);

/*
 * attn_read_prefill_skips -- synchronise `stream`, read into *skips the
 * number of prefill accesses that failed a range check since the last call on
 * this device, clear it, and return ATTN_OK if there were none,
 * ATTN_ERR_DEVICE if there were, or ATTN_ERR_CUDA.  Always 0 in release
 * builds.  `skips` may be NULL.
 */
int attn_read_prefill_skips(uint32_t* skips, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
