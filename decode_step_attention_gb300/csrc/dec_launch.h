// Internal launchers of the decode-step attention kernels (host side). Arguments
// are already validated by the C-ABI layer in api.cu; each launcher only enqueues
// its kernel and returns cudaGetLastError().
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "decattn.h"
#include "rope_angles.cuh"

namespace decattn {

// Launch `kernel` on `stream` allowing programmatic dependent launch, so that its
// launch overlaps the tail of the previous kernel (which it waits for in-kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Store a one-line reason for dec_last_error() on this thread and return `status`.
dec_status record_error(dec_status status, const char *message);

// Every host-side check dec_gqa_decode_attn makes for these arguments (shape, pointers,
// alignment, where each buffer lives, workspace size, tensor-map encoding), without
// launching anything. DEC_OK means the same call would be accepted.
dec_status attn_check(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *lens, void *out, int B, int Hq, int Hkv, int D, int T_cap,
                      int max_len, float scale, int num_parts, void *workspace,
                      size_t ws_bytes);
// DEC_OK when plain loads and stores of the kernels can reach p (device memory, or
// page-locked host memory mapped at the same address) or p is null.
dec_status check_reachable(const void *p, const char *name);


cudaError_t launch_rmsnorm_residual(const void *x, void *residual, const void *weight, void *y,
                                    int B, int hidden, float eps, cudaStream_t stream);

// K2 reading q (sequence stride q_stride elements) and new K/V (stride kv_stride) from
// anywhere, e.g. the column blocks of a packed QKV projection; rotated q to q_out.
cudaError_t launch_qknorm_rope_append_strided(const void *q_in, void *q_out, size_t q_stride,
                                              const void *k_new, const void *v_new,
                                              size_t kv_stride, const void *q_norm_w,
                                              const void *k_norm_w, void *k_cache, void *v_cache,
                                              const int32_t *pos, int B, int Hq, int Hkv, int D,
                                              int T_cap, const InvFreq &inv, int interleaved,
                                              float eps, uint32_t *error_word,
                                              cudaStream_t stream);

// Projection y = x W^T (+ residual) on the tensor cores. wmap: W [N, K] bf16, box 64 x
// 128, 128-byte swizzle; xmap: x [B, K] bf16, box 64 x plan.nb, same swizzle. A plan is
// the batch tile nb (rows of x per CTA, the MMA's N: 16 .. 256) and the K split
// (`splits` CTAs, a cluster, share each output tile, one K slice each).
struct LinPlan {
  int nb, splits;
};
int linear_batch_tile(int B);  // the smallest tile that holds B rows (at most 256)
// The plan of lowest modelled cost on `device` (forced_splits > 0: that K split, made
// even so that no slice is empty). Without a device to ask, linear_batch_tile(B) and one
// slice.
LinPlan linear_plan(int B, int N, int K, int device, bool norm = false, int forced_splits = 0);

// Epilogue of the packed QKV projection with head_dim 128 (one head per 128-feature
// tile): per-head QK-RMSNorm and RoPE at pos[b], rotated q to q_out [B, Hq, 128], K and V
// into cache slot pos[b] (see qknorm_rope_append.cu for the same step on its own).
struct QkvRotArgs {
  void *q_out, *k_cache, *v_cache;
  const int32_t *pos;
  const void *q_norm_w, *k_norm_w;  // both null: no QK-norm
  int Hq, Hkv, T_cap, interleaved;
  float eps;
  unsigned long long turns[64];  // rope angles per position, see rope_angles.cuh
};
// The RMSNorm prologue of a projection: the operand is RMSNorm(x + r) of the block's
// step (1), formed tile by tile inside the projection instead of by its own launch.
// xmap / rmap: x and r [B, K] bf16 with the operand's box; r may be absent (has_r = 0,
// the sum is x alone). The projection runs on u = bf16((x + r) * norm_w) and each batch
// row's accumulator is scaled by rsqrt(mean_K((x + r)^2) + eps) in the epilogue (the
// sums of squares of a split K are added across the cluster). h_out (optional) gets
// bf16(x + r), written once by the CTAs of the first feature tile.
struct LinNorm {
  const void *norm_w;  // [K] bf16
  void *h_out;         // [B, K] bf16 or null
  float inv_k, eps;
  int has_r;
};
cudaError_t launch_linear_qkv_rot(const CUtensorMap &wmap, const CUtensorMap &xmap, int B,
                                  int N, int K, const LinPlan &plan, const QkvRotArgs &rot,
                                  uint32_t *error_word, cudaStream_t stream,
                                  const CUtensorMap *rmap = nullptr,
                                  const LinNorm *norm = nullptr);
cudaError_t launch_linear(const CUtensorMap &wmap, const CUtensorMap &xmap, const void *residual,
                          void *y, int B, int N, int K, const LinPlan &plan,
                          uint32_t *error_word, cudaStream_t stream);
cudaError_t launch_linear_norm(const CUtensorMap &wmap, const CUtensorMap &xmap,
                               const CUtensorMap &rmap, const LinNorm &norm, void *y, int B,
                               int N, int K, const LinPlan &plan, uint32_t *error_word,
                               cudaStream_t stream);

// The whole decode step in one launch for short contexts (decode_small.cu): K1, K2,
// and the attention split over `splits` CTAs of a cluster per (sequence, KV head) with
// the merge inside the cluster. small_step_splits: the split it uses for this shape, 0
// when the shape is left to the three-launch path (more than kSmallMaxRows attended
// rows, more than kSmallMaxPairs (sequence, KV head) pairs, or more than 8 query heads
// per KV head).
constexpr int kSmallMaxRows = 1024;
constexpr int kSmallMaxPairs = 64;
int small_step_splits(int B, int Hq, int Hkv, int D, int max_len, int window);
cudaError_t launch_decode_small(const void *x, void *residual, const void *norm_w, void *y,
                                int hidden, float eps, void *q, const void *k_new,
                                const void *v_new, const void *q_norm_w, const void *k_norm_w,
                                void *k_cache, void *v_cache, const int32_t *pos,
                                const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                                int T_cap, int splits, int window, float scale_log2,
                                const InvFreq &inv, int interleaved, uint32_t *error_word,
                                cudaStream_t stream);

// The attention call alone (q rotated, the cache appended) on the same kernel, for the
// shapes small_step_splits accepts: the split and its merge in one launch; only `out`
// (and error bits) are written.
cudaError_t launch_attn_small(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                              int T_cap, int splits, int window, float scale_log2,
                              uint32_t *error_word, cudaStream_t stream);

// The fused sampler: one cluster of CTAs per row of logits (sampler_cluster(V) for a
// few rows), each holding its slice in shared memory (at most kSamplerMaxSmem).
// sampler_supports: whether a row of V logits fits a cluster of 16.
constexpr size_t kSamplerMaxSmem = 200 * 1024;
int sampler_cluster(int V);
bool sampler_supports(int V);
cudaError_t launch_sampler(const float *logits, const int32_t *ids, int L, const float *u,
                           int32_t *tokens, int B, int V, float penalty, float temperature,
                           float top_p, int top_k, cudaStream_t stream);

// K1 and K2 of one decode step in one launch (arguments as the two calls).
cudaError_t launch_rms_rope_fused(const void *x, void *residual, const void *norm_w, void *y,
                                  int hidden, float eps, void *q, const void *k_new,
                                  const void *v_new, const void *q_norm_w, const void *k_norm_w,
                                  void *k_cache, void *v_cache, const int32_t *pos, int B, int Hq,
                                  int Hkv, int D, int T_cap, const InvFreq &inv, int interleaved,
                                  uint32_t *error_word, cudaStream_t stream);

// Split pass geometry: pipeline stages that fit the device's shared memory for this
// shape (0 if none), and the dynamic shared memory that many stages take.
int split_stages(int D, int G, int B, int device);
size_t split_smem_bytes(int D, int G, int B, int stages);

// kmap/vmap: boxes of 64 dims x kSplitBoxRows tokens; kmap8/vmap8: 64 dims x 8 tokens.
// fused: the split pass and its merge in one cooperative launch (out_direct receives
// every head; max_len sizes the merge's warps per head); it needs split_fused_fits.
cudaError_t launch_gqa_split(const CUtensorMap &kmap, const CUtensorMap &vmap,
                             const CUtensorMap &kmap8, const CUtensorMap &vmap8, const void *q,
                             const int32_t *lens, int B, int Hq, int Hkv, int D, int T_cap,
                             float scale_log2, int num_parts, void *workspace, void *out_direct,
                             int window, cudaStream_t stream, bool fused = false,
                             int max_len = 0);
// Whether num_parts CTAs of the split pass can all be resident at once on `device`
// (one per SM; the device supports cooperative launches): the one-launch attention.
bool split_fused_fits(int num_parts, int device);

cudaError_t launch_split_merge(const void *workspace, void *out, int B, int Hq, int Hkv, int D,
                               int max_len, int num_parts, cudaStream_t stream);

}  // namespace decattn
