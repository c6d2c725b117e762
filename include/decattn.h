/*
 * decattn.h — C ABI of libdecattn.so, the decode-step attention block for sm_103a.
 *
 * The block is the per-token attention step of a dense RoPE + RMSNorm + GQA decoder:
 *   (1) RMSNorm with a fused residual add,
 *   (2) per-head QK-RMSNorm, RoPE (NeoX or interleaved) at a per-sequence position,
 *       and the bf16 K/V append into a contiguous KV cache,
 *   (3) single-query GQA attention over that cache with an online softmax, a
 *       split-KV pass and a log-sum-exp merge, with per-sequence lengths.
 * Sources: fusedtok 1.0.1 README ("Operators" table, "Usage", "Benchmarks");
 * cutileGPT README ("Why tiles", "The current runtime includes").
 *
 * Conventions for every entry point
 *   - Pointers marked [device] are CUDA device pointers on the current device,
 *     16-byte aligned, owned by the caller. The library allocates, frees and
 *     synchronises nothing, and keeps no state apart from a per-device cache of
 *     the SM count and kernel attributes.
 *   - Pointers marked [device|host] may also point into page-locked host memory
 *     that is mapped into the device's address space at the same address (memory
 *     from cudaHostAlloc / cudaMallocHost under unified addressing). The kernels
 *     then read or write it across the host link themselves, with no copy step: a
 *     host-to-host step needs no cudaMemcpy around it. Before launching, every call
 *     asks the runtime where each pointer lives (cudaPointerGetAttributes) and
 *     refuses with DEC_ERR_INVALID_ARG one the kernels could not reach: pageable
 *     host memory, or host memory for a [device] argument (those are read with
 *     bulk-tensor or bulk copies, which are only given device memory).
 *   - bf16 tensors are IEEE bfloat16, row-major and contiguous in the shape given.
 *     Arithmetic is fp32 inside the kernels; results are rounded to bf16 (RNE)
 *     once, at the store.
 *   - Every call only enqueues work on `stream` (0 = legacy default stream) and
 *     returns. Arguments are checked on the host first: a failed check returns a
 *     non-zero status and launches nothing. A launch failure returns
 *     DEC_ERR_CUDA. dec_last_error() gives a one-line reason for the last
 *     non-zero status on the calling thread.
 *   - Lengths and positions live on the device and cannot be checked by the host.
 *     Kernels clamp a length to [0, T_cap] and skip a position outside
 *     [0, T_cap), raising a bit in a device error word (see DEC_DEVERR_*).
 *   - Re-entrant; calls on different streams may overlap if their buffers do not.
 *   - Every kernel is launched with programmatic dependent launch: it may start while
 *     the kernel before it on the stream finishes, and waits for that kernel before it
 *     reads anything the kernel could have written. Only this library's kernels let a
 *     successor start early, and none of them writes a length array or a projection
 *     weight, so the attention kernels read `lens` (and prefetch their first cache
 *     tiles into L2), and the projections request their first weight tiles, before
 *     that wait. Anything else a call reads or writes waits for it.
 */
#ifndef DECATTN_H_
#define DECATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *dec_stream_t;

typedef enum dec_status {
  DEC_OK = 0,
  DEC_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad size or shape */
  DEC_ERR_UNSUPPORTED = 2,  /* a valid shape the library has no kernel for */
  DEC_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  DEC_ERR_CUDA = 4          /* the CUDA runtime or driver reported an error */
} dec_status;

typedef enum dec_rope_layout {
  DEC_ROPE_NEOX = 0,        /* element i pairs with i + D/2 */
  DEC_ROPE_INTERLEAVED = 1  /* element 2i pairs with 2i + 1 */
} dec_rope_layout;

/* RoPE frequency tables for context extension (PyGPUkit 0.2.18 page, "Positional
 * Encoding Operations": rope_init_linear, rope_init_ntk_aware; the page names them
 * without formulas). With s the factor:
 *   DEC_ROPE_SCALE_NONE    inv_freq_i = theta^(-2i/D)
 *   DEC_ROPE_SCALE_LINEAR  inv_freq_i = theta^(-2i/D) / s      (positions divided by s)
 *   DEC_ROPE_SCALE_NTK     inv_freq_i = (theta * s^(D/(D-2)))^(-2i/D): the base grows so
 *                          that pair 0 keeps frequency 1 and the slowest pair turns s
 *                          times slower. */
typedef enum dec_rope_scaling {
  DEC_ROPE_SCALE_NONE = 0,
  DEC_ROPE_SCALE_LINEAR = 1,
  DEC_ROPE_SCALE_NTK = 2
} dec_rope_scaling;

/* Fills inv_freq[0 .. D/2) (host memory, owned by the caller) with the table above, in
 * fp64. D in {64, 128}; rope_theta finite, > 0; factor finite, >= 1 (not read for
 * DEC_ROPE_SCALE_NONE). Host only: launches nothing and needs no device. The table, or
 * any other with D/2 entries in [0, 1], goes to the rotating calls below as their
 * `inv_freq` argument. */
dec_status dec_rope_inv_freq(int D, float rope_theta, dec_rope_scaling scaling, float factor,
                             double *inv_freq);

/* The YaRN table (PyGPUkit 0.2.18 page, "Positional Encoding Operations":
 * rope_init_yarn, named only; the published YaRN method). Pair i of the plain table, with
 * frequency f_i = theta^(-2i/D), turns r_i = original_context * f_i / (2 pi) times over
 * the original context; it keeps f_i where r_i >= beta, takes f_i / s where r_i <= alpha,
 * and (1 - g) f_i / s + g f_i with g = (r_i - alpha) / (beta - alpha) between (s = the
 * factor). The method also multiplies the rotated q and k by m = 0.1 ln(s) + 1; here
 * that temperature is carried by the softmax scale instead, which gives the same
 * attention while the cache keeps unscaled keys: *scale_mult (optional) receives m^2,
 * and the attention calls take scale = m^2 / sqrt(D).
 * D in {64, 128}; rope_theta finite, > 0; factor finite, >= 1; original_context >= 1;
 * 0 <= alpha < beta (the method's values for Llama-family models: 1 and 32).
 * inv_freq: host double [D/2], owned by the caller. Host only. */
dec_status dec_rope_yarn_inv_freq(int D, float rope_theta, float factor, int original_context,
                                  float alpha, float beta, double *inv_freq,
                                  float *scale_mult);
/* The softmax scale that carries YaRN's temperature for head_dim D, m^2 / sqrt(D) with m =
 * 0.1 ln(factor) + 1, into *scale (host). factor finite, >= 1. Host only. */
dec_status dec_rope_yarn_softmax_scale(int D, float factor, float *scale);

/* Bits of the device error word (first 4 bytes of the attention workspace, or
 * the optional error word given to dec_qknorm_rope_kv_append). Set with atomicOr,
 * never cleared by the library. */
#define DEC_DEVERR_LEN_CLAMPED   0x1u  /* a lens[b] outside [0, T_cap] was clamped */
#define DEC_DEVERR_POS_SKIPPED   0x2u  /* a pos[b] outside [0, T_cap) was skipped */
#define DEC_DEVERR_WAIT_TIMEOUT  0x4u  /* a pipeline wait gave up (results invalid) */

/* ------------------------------------------------------------------------ K1
 * RMSNorm with a fused residual add (fusedtok README, "Operators": RMSNorm
 * (+residual); "Usage": h = rmsnorm(h, w, residual=h); cutileGPT README, "Why
 * tiles": rstd = 1/sqrt(sum(x*x)/N + eps), y = x*rstd*w).
 *
 *   s        = x + residual          (fp32; residual omitted when NULL)
 *   residual = bf16(s)               (written back when residual != NULL)
 *   y        = bf16(s * rsqrt(mean(s^2) + eps) * weight)   (from the fp32 s)
 *
 * x, y      [device|host] bf16 [B, hidden];  y may not alias x or residual.
 * residual  [device|host] bf16 [B, hidden], read then overwritten; or NULL.
 * weight    [device|host] bf16 [hidden].
 * hidden    multiple of 8, 8 .. 16384.  B >= 0 (B == 0 launches nothing).
 * eps       >= 0.
 */
dec_status dec_rmsnorm_residual(const void *x, void *residual, const void *weight, void *y,
                                int B, int hidden, float eps, dec_stream_t stream);

/* ------------------------------------------------------------------------ K2
 * Per-head QK-RMSNorm, RoPE and the K/V append (cutileGPT README, "The current
 * runtime includes": fused QK-Norm + RoPE + KV-cache writes; fusedtok README,
 * "Operators": RoPE in interleaved and NeoX layouts with a kv-cache position
 * offset; "Usage": rope(q, pos_offset=..., neox=True), caches [B, Hkv, T, D]).
 *
 * For sequence b at position p = pos[b] and every head:
 *   u   = RMSNorm_D(head, norm weight, eps)   (skipped when the weight is NULL)
 *   out = RoPE(u, p): pair (a, b) -> (a cos f - b sin f, a sin f + b cos f),
 *         f = p * inv_freq_i for pair i (angles formed in fp64), inv_freq_i =
 *         theta^(-2i/D), or the caller's table.
 *   q[b, h]               <- bf16(out)       (in place)
 *   k_cache[b, g, p, :]   <- bf16(out of k_new[b, g])
 *   v_cache[b, g, p, :]   <- v_new[b, g]     (bit copy)
 * Other cache slots are untouched. A pos[b] outside [0, T_cap) skips sequence b
 * (its q is left as is) and raises DEC_DEVERR_POS_SKIPPED in *error_word.
 *
 * q          [device|host] bf16 [B, Hq, D], in/out.
 * k_new      [device|host] bf16 [B, Hkv, D];  v_new [device|host] bf16 [B, Hkv, D].
 * q_norm_w, k_norm_w  [device|host] bf16 [D] each, or both NULL (QK-norm off).
 * k_cache, v_cache    [device] bf16 [B, Hkv, T_cap, D].
 * pos        [device|host] int32 [B].
 * error_word [device|host] uint32, or NULL.
 * inv_freq   [host] double [D/2], each in [0, 1], read during the call (a graph
 *            captured from the call keeps the values); or NULL for theta^(-2i/D), in
 *            which case rope_theta must be finite and > 0 (it is not read otherwise).
 *            Every call below that rotates takes the same argument.
 * D in {64, 128}; Hq % Hkv == 0.
 */
dec_status dec_qknorm_rope_kv_append(void *q, const void *k_new, const void *v_new,
                                     const void *q_norm_w, const void *k_norm_w,
                                     void *k_cache, void *v_cache, const int32_t *pos,
                                     int B, int Hq, int Hkv, int D, int T_cap,
                                     float rope_theta, dec_rope_layout layout,
                                     const double *inv_freq, float eps,
                                     uint32_t *error_word, dec_stream_t stream);

/* As dec_qknorm_rope_kv_append, but q is read from q_in and the rotated q written
 * to q_out (q_in itself is left as is; a skipped sequence's q_out is left as is).
 * q_in and q_out are the same buffer or do not overlap. With q_in in mapped host
 * memory and q_out on the device, the query of a host-staged step goes straight
 * into the buffer the attention call reads.
 * q_in [device|host], q_out [device|host] bf16 [B, Hq, D]; the rest as above. */
dec_status dec_qknorm_rope_kv_append_out(const void *q_in, void *q_out, const void *k_new,
                                         const void *v_new, const void *q_norm_w,
                                         const void *k_norm_w, void *k_cache, void *v_cache,
                                         const int32_t *pos, int B, int Hq, int Hkv, int D,
                                         int T_cap, float rope_theta, dec_rope_layout layout,
                                         const double *inv_freq, float eps,
                                         uint32_t *error_word, dec_stream_t stream);

/* ------------------------------------------------------------------ K3 + K4
 * Single-query GQA decode attention over a contiguous cache (fusedtok README,
 * "Operators": attention_decode — online softmax, flash-decoding split over long
 * caches, per-sequence lengths; "Usage": q [B, Hq, D], caches [B, Hkv, T, D],
 * lens [B] int32; "Benchmarks": heads expanded with repeat_interleave, so query
 * head h reads KV head h / (Hq/Hkv)).
 *
 *   out[b, h] = sum_{t < lens[b]} softmax_t(scale * q[b,h] . K[b,g,t]) V[b,g,t],
 *   g = h / (Hq/Hkv).  A sequence with lens[b] == 0 gives zeros.
 *
 * Split pass (K3, `num_parts` CTAs, one per SM by default): the Hkv * sum_b lens[b]
 * (sequence, KV head, token) rows are read as one stream and cut into num_parts
 * blocks of blk = max(64, ceil(rows/num_parts)) rows. A block of at least 4096 rows
 * is one piece of floor(4*blk/5) rows, taken by its own CTA, followed by 4 pieces of
 * ceil((blk - floor(4*blk/5))/4) rows that CTAs claim from a counter as they finish;
 * a smaller block is a single piece.
 * A piece that crosses a (sequence, KV head) boundary yields one partial per pair
 * it touches. Each CTA serves the whole GQA group of a KV head from one read of
 * each K/V tile. A partial holds, for each of the G query heads, the normalised o
 * (fp32 [D]) and lse in base 2 (log2 sum 2^(scale*log2(e)*s)). Results do not
 * depend on which CTA claims which piece.
 * Merge pass (K4): out = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M).
 * dec_gqa_decode_attn lets the split pass write out[b, h] itself (normalised, bf16)
 * for every (b, g) pair whose rows lie in a single piece; the merge fills in the
 * others (the flag at byte 12 of the workspace says which mode the last split pass
 * ran in). dec_gqa_decode_split alone always writes partials.
 * When num_parts is at most the SM count (always so with num_parts = 0),
 * dec_gqa_decode_attn and dec_gqa_decode_attn_window run the split pass and the merge
 * as ONE cooperative launch (every CTA resident at once): each CTA marks its pieces
 * done as it finishes them, and then merges its share of the query heads, each as soon
 * as the pieces of its pair are marked (the waits are bounded in time like the
 * pipeline waits). The marks carry a launch epoch kept in the header (byte 28, one
 * more after every such call), so marks left by earlier calls never count.
 * Short contexts: with num_parts = 0 and a shape for which dec_decode_step_launches
 * reports 1 (at most 1024 attended rows, at most 64 (sequence, KV head) pairs),
 * dec_gqa_decode_attn and dec_gqa_decode_attn_window run as ONE launch instead: the
 * rows of each pair are split over a cluster of up to 8 CTAs whose softmax states
 * merge in distributed shared memory. Only out and the error word are written then.
 *
 * Workspace layout ([device], caller-allocated, at least
 * dec_attn_workspace_bytes(...) bytes, 256-byte aligned): a 256-byte header — a
 * uint32 device error word at byte 0, two uint32 claim counters at bytes 4 and 8
 * (zero before the first use, back at zero after every completed split pass; after a
 * DEC_DEVERR_WAIT_TIMEOUT, zero the whole workspace again before its next use) and
 * the direct-output flag at byte 12 — then the o partials fp32 [S][G][D] at byte 256, then the
 * lse partials fp32 [S][G], S = 5*num_parts + B*Hkv, then (16-byte aligned) the
 * sequence offsets int32 [B+1] (exclusive prefix sums of the clamped lengths) that
 * the split pass writes and the merge pass reads, then (16-byte aligned) one uint32
 * completion mark per piece [5*num_parts]. The whole workspace is zeroed before its
 * first use. Partials of pair p from piece i
 * sit in slot i + p. One workspace serves one call at a time; dec_split_merge
 * merges what the last split pass on that workspace left there (its `lens` must be
 * the array that pass was given; the offsets are read from the workspace).
 *
 * q          [device] bf16 [B, Hq, D] (already rotated).
 * k_cache, v_cache [device] bf16 [B, Hkv, T_cap, D]; rows t >= lens[b] may hold
 *            anything (NaN included): they are never used.
 * lens       [device|host] int32 [B].
 * out        [device|host] bf16 [B, Hq, D].
 * max_len    host upper bound of every lens[b] (sizes the grid; 0 <= max_len <= T_cap).
 * scale      softmax scale; <= 0 selects 1/sqrt(D).
 * num_parts  CTAs of the split pass; 0 selects dec_attn_default_parts(). The
 *            merge must be given the same value as the split pass.
 * D in {64, 128}; 1 <= Hq/Hkv <= 8; B*Hkv*max_len < 2^31; B <= 16384.
 */
int dec_attn_default_parts(int B, int Hkv, int D, int max_len);
size_t dec_attn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len, int num_parts);

/* The two sizing helpers under the names of the block's interface statement (fusedtok
 * README, "Operators": attention_decode with a flash-decoding split over long caches;
 * "Usage": caller-owned tensors, stream-ordered calls). Here a "split" is one CTA of
 * the split pass: the stream of (sequence, KV head, token) rows is cut into that many
 * blocks, not each sequence into that many chunks, so the count depends on the total
 * rows and the SM count rather than on one sequence's length. Host only.
 *   dec_pick_num_splits: the num_parts the library picks for the split pass, min(sm_count,
 *     ceil(B * Hkv * max_len / 64)), at least 1; sm_count <= 0 reads the current device's
 *     SM count. dec_attn_default_parts is the same with the current device's count.
 *   dec_decode_workspace_bytes: an attention workspace size that serves every split
 *     count up to max_splits (<= 0: the current device's SM count) and every KV head
 *     count Hkv that divides Hq with Hq / Hkv <= 8, at any max_len; 0 for B < 0, Hq <= 0
 *     or D outside {64, 128}. dec_attn_workspace_bytes gives the exact size of one
 *     shape. */
int dec_pick_num_splits(int B, int Hkv, int max_len, int sm_count);
size_t dec_decode_workspace_bytes(int B, int Hq, int D, int max_splits);

dec_status dec_gqa_decode_split(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *lens, int B, int Hq, int Hkv, int D, int T_cap,
                                int max_len, float scale, int num_parts, void *workspace,
                                size_t workspace_bytes, dec_stream_t stream);

dec_status dec_split_merge(const void *workspace, size_t workspace_bytes, const int32_t *lens,
                           void *out, int B, int Hq, int Hkv, int D, int T_cap, int max_len,
                           int num_parts, dec_stream_t stream);

/* Split pass then merge pass, on one stream. */
dec_status dec_gqa_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                               int T_cap, int max_len, float scale, int num_parts,
                               void *workspace, size_t workspace_bytes, dec_stream_t stream);

/* Sliding-window decode attention (cutileGPT README, "The current runtime
 * includes": sliding-window attention): as dec_gqa_decode_attn, but sequence b
 * attends only to its last min(lens[b], window) tokens, rows
 * [lens[b] - window, lens[b]) — the new token and the window-1 before it. The split
 * pass streams only those rows. window >= 1; a window >= lens[b] is plain
 * attention for that sequence. The workspace size is that of dec_gqa_decode_attn. */
dec_status dec_gqa_decode_attn_window(const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *lens, void *out, int B, int Hq, int Hkv,
                                      int D, int T_cap, int max_len, int window, float scale,
                                      int num_parts, void *workspace, size_t workspace_bytes,
                                      dec_stream_t stream);

/* ------------------------------------------------------- allocation-free
 * The attention call above with its workspace replaced by a scratch buffer the
 * library keeps in static device memory. The pages have no counterpart of this
 * call; it exists for callers that cannot allocate device memory at the point of
 * the call (a host callback or allocator hook where cudaMalloc would re-enter the
 * allocator, a plugin inside a runtime that owns every allocation, code that must
 * keep the process's memory footprint fixed). It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *   - The scratch is 4 MiB per device, held by every GPU that loads the library
 *     until the process exits. A shape whose partials need more (see
 *     dec_attn_workspace_bytes) is rejected with DEC_ERR_WORKSPACE, launching
 *     nothing.
 *   - All calls on a device share the buffer; calls whose kernels overlap on the
 *     GPU race and give wrong results. The buffer keeps the previous call's
 *     contents; each call, once every argument check has passed, first clears its
 *     header (error word and claim counters) on `stream`. A refused call enqueues
 *     nothing.
 *   - error_word [device|host] uint32, 4-byte aligned, or NULL: when given, the call
 *     copies its device error word (DEC_DEVERR_* bits; this call's alone, since the
 *     word is cleared first) there on `stream` after the kernels. The scratch itself
 *     is not readable by the caller, and the next call clears it.
 *   - Every call looks the buffer's device address up on the current device (so a
 *     reset or recreated context is followed). The first call on a device may load
 *     the module there; make that first call before any stream capture.
 * Other arguments as for dec_gqa_decode_attn.
 */
dec_status dec_gqa_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *lens, void *out, int B, int Hq, int Hkv,
                                       int D, int T_cap, int max_len, float scale, int num_parts,
                                       uint32_t *error_word, dec_stream_t stream);

/* ------------------------------------------------------------- whole block
 * K1, K2, K3 and K4 in order on one stream: the decode step of the block for
 * inputs already resident on the device. Arguments as in the calls above; the
 * projections between RMSNorm and the rotation are outside the block, so q,
 * k_new and v_new are inputs of their own, and K1 and K2 run in one launch. The
 * error word of K2 is the workspace's. window = 0 attends to the whole sequence,
 * window > 0 as dec_gqa_decode_attn_window. All arguments are checked before the
 * first launch. q is [device] here (the split pass reads the rotated q with bulk
 * copies), except on the one-launch path below, where it is [device|host] too; x,
 * residual, y, k_new, v_new, pos, lens and out are [device|host]. With
 * the inputs in mapped host memory the one fused K1 + K2 launch reads all of them
 * across the host link before the split pass can start; a host-staged step is
 * quicker as K2 (dec_qknorm_rope_kv_append_out) -> attention on one stream with K1
 * on another beside it, since K1's host traffic then overlaps the split pass.
 * Short contexts (at most 1024 attended rows, at most 64 (sequence, KV head) pairs)
 * run as ONE launch instead: K1, K2 and the attention in one kernel, the rows of each
 * (sequence, KV head) split over a cluster of up to 8 CTAs whose softmax states merge
 * in distributed shared memory; results as the three-launch path (the same roundings:
 * the stored q, K and V are what the attention uses). Longer contexts take two
 * launches: K1 + K2, then the attention's split pass and merge in one cooperative
 * launch (one CTA per SM, every CTA resident at once, each query head merged as soon as
 * its pieces are marked done), or three (the merge on its own) when num_parts exceeds
 * the SM count. dec_decode_step_path reports which form a shape takes with
 * num_parts = 0 on the current device, dec_decode_step_launches how many launches that
 * is (1, 2 or 3).
 */
typedef enum dec_step_path {
  DEC_STEP_SHORT = 0,   /* one launch: the short-context kernel (clusters, DSMEM merge) */
  DEC_STEP_STREAM = 1,  /* two launches: K1 + K2, then split pass + merge, cooperative */
  DEC_STEP_THREE = 2    /* three launches: K1 + K2, split pass, merge */
} dec_step_path;
int dec_decode_step_path(int B, int Hq, int Hkv, int D, int max_len, int window);
int dec_decode_step_launches(int B, int Hq, int Hkv, int D, int max_len, int window);
dec_status dec_decode_step(const void *x, void *residual, const void *norm_w, void *y,
                           int hidden, float eps,
                           void *q, const void *k_new, const void *v_new,
                           const void *q_norm_w, const void *k_norm_w,
                           void *k_cache, void *v_cache, const int32_t *pos,
                           const int32_t *lens, void *out,
                           int B, int Hq, int Hkv, int D, int T_cap, int max_len,
                           float rope_theta, dec_rope_layout layout, const double *inv_freq,
                           float scale, int window, int num_parts, void *workspace,
                           size_t workspace_bytes, dec_stream_t stream);

/* ------------------------------------------------------------ projections
 * y = x W^T, plus residual when given: the projections on either side of the
 * block (cutileGPT README, "The current runtime includes": packed QKV projections,
 * fused down-projection + residual epilogues; PyGPUkit 0.2.18 page, "Optimized
 * BF16 GEMV": the weight stored one row per output feature, B[N, K]).
 *
 *   x        [device] bf16 [B, K]
 *   w        [device] bf16 [N, K]     row n holds the weights of output feature n
 *   residual [device|host] bf16 [B, N]  added in fp32 before the single rounding; may
 *                                     be NULL, or be y itself (in-place add)
 *   y        [device|host] bf16 [B, N]  y[b, n] = bf16(sum_k x[b, k] w[n, k] + r[b, n]);
 *                                     must not overlap x or w
 *   k_split  0: choose the K split automatically; 1 .. min(8, K/64): use that many
 *            CTAs (one cluster) per output tile, each taking an equal K slice
 *   error_word [device|host] uint32, optional (DEC_DEVERR_WAIT_TIMEOUT)
 *   N a positive multiple of 128, K a positive multiple of 64, B >= 0 (B = 0 is a
 *   no-op). Runs on the tensor cores with fp32 accumulation, in one launch. When the
 *   output tiles alone would leave SMs idle, K is split over a cluster of up to 8
 *   CTAs per tile whose partial sums are added in a fixed order inside the cluster
 *   (distributed shared memory, no round trip through HBM), so results are
 *   identical from run to run on the same device.
 * dec_linear_plan reports the batch tile (16 .. 256 rows) and the K split
 * dec_linear chooses for this shape on the current device.
 */
dec_status dec_linear_plan(int B, int N, int K, int *batch_tile, int *k_split);
dec_status dec_linear(const void *x, const void *w, const void *residual, void *y,
                      int B, int N, int K, int k_split, uint32_t *error_word,
                      dec_stream_t stream);

/* The packed QKV projection with the rotation step as its epilogue (cutileGPT
 * README, "The current runtime includes": packed QKV projections, fused QK-Norm +
 * RoPE + KV-cache writes), head_dim 128 only: [q | k | v] = y w_qkv^T is not stored;
 * per head and sequence b the projected q and k get the QK-RMSNorm (when the weights
 * are given) and RoPE at pos[b] as in dec_qknorm_rope_kv_append, q goes to q_out
 * [B, Hq, 128] and k and v to cache slot pos[b].
 *   y [device] bf16 [B, hidden]; w_qkv [device] bf16 [(Hq + 2 Hkv) 128, hidden]
 *   (columns: q heads, k heads, v heads); other arguments as dec_qknorm_rope_kv_append
 *   (q_out [device|host]); error_word [device|host] uint32, optional. hidden a
 *   positive multiple of 64.
 */
dec_status dec_qkv_proj_rope_append(const void *y, const void *w_qkv, const void *q_norm_w,
                                    const void *k_norm_w, void *q_out, void *k_cache,
                                    void *v_cache, const int32_t *pos, int B, int hidden,
                                    int Hq, int Hkv, int D, int T_cap, float rope_theta,
                                    dec_rope_layout layout, const double *inv_freq, float eps,
                                    uint32_t *error_word, dec_stream_t stream);

/* Projections with the RMSNorm of step (1) as their prologue (cutileGPT README, "The
 * current runtime includes": packed QKV projections, RMSNorm; fusedtok README,
 * "Operators": RMSNorm (+residual), fusion to cut global-memory round trips). Instead of a
 * separate RMSNorm launch and a round trip of y through memory, the projection forms
 * its operand from x and the residual tile by tile:
 *   s = x + residual (fp32; residual NULL: s = x),  h = bf16(s)
 *   u = bf16(s * norm_w)                 (the tensor-core operand)
 *   y[b, n] = rsqrt(mean_k s[b, k]^2 + eps) * sum_k u[b, k] w[n, k]
 * i.e. RMSNorm(h) w^T with the row scale applied to the fp32 accumulator; every
 * value is rounded to bf16 once, as in the unfused pair (RMSNorm output, then the
 * projection), and both agree with the exact result to the same bound.
 *   x, residual [device] bf16 [B, K] (read with bulk-tensor copies); residual may be NULL.
 *   norm_w      [device] bf16 [K] (read with bulk copies).
 *   h_out       [device|host] bf16 [B, K] or NULL: receives h. It may not overlap x,
 *               residual or the output (other CTAs still read x and residual), so an
 *               in-place residual update is the caller's next step.
 *   eps >= 0; the rest as dec_linear (N a multiple of 128, K of 64).
 * dec_norm_linear: y [device|host] bf16 [B, N] = RMSNorm(x + residual) w^T.
 * dec_norm_qkv_proj_rope_append: the packed QKV projection of RMSNorm(x + residual)
 * with the rotation epilogue of dec_qkv_proj_rope_append (head_dim 128; eps serves
 * both norms).
 * Cost: every feature tile forms the operand again from x and the residual. At decode
 * batches (up to 64 rows) that is about the cost of the separate RMSNorm launch it
 * replaces; at larger batches the separate launch is cheaper, and the attention
 * sublayer below keeps it. */
dec_status dec_norm_linear(const void *x, const void *residual, const void *norm_w, void *h_out,
                           const void *w, void *y, int B, int N, int K, float eps, int k_split,
                           uint32_t *error_word, dec_stream_t stream);
dec_status dec_norm_qkv_proj_rope_append(const void *x, const void *residual,
                                         const void *norm_w, void *h_out, const void *w_qkv,
                                         const void *q_norm_w, const void *k_norm_w,
                                         void *q_out, void *k_cache, void *v_cache,
                                         const int32_t *pos, int B, int hidden, int Hq, int Hkv,
                                         int D, int T_cap, float rope_theta,
                                         dec_rope_layout layout, const double *inv_freq,
                                         float eps, uint32_t *error_word, dec_stream_t stream);

/* ------------------------------------------------------ attention sublayer
 * The attention half of one decoder layer around the block, on one stream:
 *
 *   h          = x + residual        (residual buffer <- bf16(h); h = x when NULL)
 *   y          = RMSNorm(h) * norm_w
 *   [q | k | v] = y w_qkv^T           packed projection, columns: Hq q heads, then
 *                                    Hkv k heads, then Hkv v heads, D each
 *   q, k       <- QK-norm + RoPE at pos[b]; k and v written to cache slot pos[b]
 *   a          = attention of q over the cache (window as dec_decode_step)
 *   out        = bf16(h + a w_o^T)
 *
 *   w_qkv [device] bf16 [(Hq + 2 Hkv) D, hidden];  w_o [device] bf16 [hidden, Hq D]
 *   out   [device|host] bf16 [B, hidden], must not overlap x or residual.
 *   x, residual, norm_w, pos, lens [device|host]; the caches and the workspace [device].
 *   Other arguments as dec_decode_step. hidden a multiple of 128 (<= 16384) and
 *   (Hq + 2 Hkv) D a multiple of 128. The intermediates (y, the packed qkv, rotated
 *   q, attention rows) live in the workspace: 256-byte
 *   aligned, at least dec_attn_sublayer_workspace_bytes, zeroed before first use;
 *   its first word is the device error word. Launches: RMSNorm, the QKV projection
 *   with the rotation as its epilogue (head_dim 128; head_dim 64: the projection, then
 *   the rotation), split pass, merge (one launch for both in the short-context case of
 *   dec_gqa_decode_attn, when num_parts = 0), output projection. With head_dim 128 the packed
 *   qkv is not stored (its workspace view is left untouched).
 */
size_t dec_attn_sublayer_workspace_bytes(int B, int hidden, int Hq, int Hkv, int D,
                                         int max_len, int num_parts);
/* Where the intermediates sit in that workspace, for inspection after the call:
 * offsets[0..4] (host array of 5) = byte offsets of y [B, hidden], the packed qkv
 * [B, (Hq + 2 Hkv) D], rotated q [B, Hq, D] and the attention rows [B, Hq, D] (all
 * bf16), and the total size. The attention workspace
 * (error word, partials) occupies [0, offsets[0]). */
dec_status dec_attn_sublayer_layout(int B, int hidden, int Hq, int Hkv, int D, int max_len,
                                    int num_parts, size_t *offsets);
dec_status dec_attn_sublayer(const void *x, void *residual, const void *norm_w, int hidden,
                             float eps, const void *w_qkv, const void *w_o,
                             const void *q_norm_w, const void *k_norm_w,
                             void *k_cache, void *v_cache, const int32_t *pos,
                             const int32_t *lens, void *out,
                             int B, int Hq, int Hkv, int D, int T_cap, int max_len,
                             float rope_theta, dec_rope_layout layout,
                             const double *inv_freq, float scale, int window, int num_parts,
                             void *workspace, size_t workspace_bytes, dec_stream_t stream);

/* ------------------------------------------------------------------ sampler
 * The sampling side of a decode step, fused into one launch (fusedtok README,
 * "Operators": repetition penalty, temperature, argmax, sample_topk, sample_topp,
 * decode_step = penalty -> temperature -> nucleus sample; "Usage"). Per row b:
 *   1. CTRL repetition penalty: each distinct id of sampled_ids[b, 0..L) inside
 *      [0, V) has its logit divided by `penalty` if positive, else multiplied by it
 *      (negative ids are padding; penalty 1 is a no-op);
 *   2. temperature <= 0: tokens[b] = argmax (lowest id among equal maxima), done;
 *   3. otherwise p = softmax(z / temperature);
 *   4. top_k > 0: keep the k most probable tokens (equal probabilities ranked by
 *      lowest id); 0 keeps all;
 *   5. top_p < 1: within those, keep the shortest prefix of the ranking whose mass,
 *      renormalised over the kept tokens, reaches top_p;
 *   6. draw: with the uniform u[b] in [0, 1), tokens[b] = the first kept token, in
 *      token-id order, whose running mass exceeds u[b] times the kept mass.
 * Masses are summed as 64-bit fixed point (units of 2^-40 of the largest
 * probability), so the result does not depend on summation order and is identical
 * from run to run.
 *   logits      [device|host] fp32 [B, V], finite (or -inf) with a finite maximum
 *   sampled_ids [device|host] int32 [B, L], may be NULL when L = 0
 *   u           [device|host] fp32 [B] in [0, 1) (the random numbers; NULL when greedy)
 *   tokens      [device|host] int32 [B] (output)
 *   0 <= B <= 65535; 1 <= V <= 262144; penalty > 0; top_p in (0, 1]; top_k >= 0.
 * A few rows are spread over up to 16 CTAs each (a cluster) for latency; many rows use
 * the cluster size that keeps the most rows resident at once.
 */
dec_status dec_sample(const float *logits, const int32_t *sampled_ids, int L, const float *u,
                      int32_t *tokens, int B, int V, float penalty, float temperature,
                      float top_p, int top_k, dec_stream_t stream);

/* -------------------------------------------------------------- diagnostics
 * Runs one warp that waits on a barrier nobody arrives at, with the same bounded
 * wait the pipelined kernels use, and raises DEC_DEVERR_WAIT_TIMEOUT in
 * *error_word ([device] uint32) when the wait gives up (after one second of
 * wall-clock time). Shows how a stalled pipeline is reported: an error bit, no
 * hang, the context stays usable.
 */
dec_status dec_diag_wait_timeout(uint32_t *error_word, dec_stream_t stream);

/* ------------------------------------------------------------------ helpers */
const char *dec_status_string(dec_status status);
const char *dec_last_error(void);   /* thread-local; "" after a DEC_OK call */
int dec_version(void);              /* 100 * major + minor */

#ifdef __cplusplus
}
#endif
#endif /* DECATTN_H_ */
