// K2: per-head QK-RMSNorm, RoPE at the sequence's position, and the K/V append.
//
// cutileGPT README, "The current runtime includes" (fused QK-Norm + RoPE +
// KV-cache writes); fusedtok README, "Operators" (RoPE, interleaved and NeoX
// layouts, kv-cache pos_offset) and "Usage" (rope(q, pos_offset=1023, neox=True);
// caches [B, Hkv, T, D]).
//
// A CTA handles up to 32 heads of one sequence, its eight warps taking up to four heads
// each (grid B x ceil((Hq+Hkv)/(8*hpw))): one CTA per sequence where it fits. The D/2
// rotation angles of position p are shared by every head of the sequence; each CTA
// forms them once: phi_i = p * inv_freq_i, taken as a fraction of a turn in 64-bit
// integer arithmetic (inv_freq_i / 2 pi arrives from the host as a 64-bit binary
// fraction; the whole turns fall off the top), then sin/cos in fp32 (rope_angles.cuh).
// At p ~ 1.3e5 an fp32 product would already be off by ~1e-2 rad. One warp per head: load the
// head (D/32 elements per lane), optional RMSNorm over D with a warp reduction,
// rotate (NeoX partners sit 16 lanes apart, interleaved partners in the same lane),
// store q in place or K into slot p, and copy V into slot p.
#include <math.h>

#include "dec_device.cuh"
#include "dec_launch.h"
#include "rmsnorm_body.cuh"
#include "rope_angles.cuh"
#include "rotate_head.cuh"

namespace decattn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxHeadsPerWarp = 4;

// Heads each warp of a rotation CTA takes: one while the grid stays within about two
// CTAs per SM (small batches keep their parallelism), else the fewest (at most four)
// that bring it there: fewer CTAs to launch and fewer angle tables formed again.
inline int heads_per_warp(int B, int Hq, int Hkv) {
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int h = 1;
  while (h < kMaxHeadsPerWarp &&
         (long long)B * ((Hq + Hkv + kWarps * h - 1) / (kWarps * h)) > 2LL * sms)
    ++h;
  return h;
}

// One CTA of the rotation: sequence b, the heads (q heads first, then KV heads)
// task_block*8*hpw .. +8*hpw-1, warp w taking heads w, w + 8, ... of them. The heads are
// loaded before the angle table is formed so the two latencies overlap.
// Row strides: sequence b's q heads start at q_in + b * q_stride, its new K and V heads
// at k_new / v_new + b * kv_stride (contiguous tensors, or the q / k / v column blocks of
// a packed QKV projection). Rotated q heads go to q_out [B, Hq, D], which may be q_in.
template <int D>
__device__ __forceinline__ void qknorm_rope_block(
    const __nv_bfloat16 *q_in, __nv_bfloat16 *q_out, const __nv_bfloat16 *__restrict__ k_new,
    const __nv_bfloat16 *__restrict__ v_new, const __nv_bfloat16 *__restrict__ q_norm_w,
    const __nv_bfloat16 *__restrict__ k_norm_w, __nv_bfloat16 *__restrict__ k_cache,
    __nv_bfloat16 *__restrict__ v_cache, const int32_t *__restrict__ pos, int Hq, int Hkv,
    int T_cap, size_t q_stride, size_t kv_stride, const InvFreq &inv, const RopeTurns &turns,
    int interleaved, float eps, uint32_t *error_word, int b, int task_block, int hpw,
    float *s_cos, float *s_sin) {
  using L = Lanes<D>;
  constexpr int E = L::kE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = lane * E;  // first element of this lane
  float x[kMaxHeadsPerWarp][E], w[kMaxHeadsPerWarp][E];
#pragma unroll
  for (int k = 0; k < kMaxHeadsPerWarp; ++k) {  // every head's load in flight at once
    const int task = (task_block * hpw + k) * kWarps + warp;
    if (k < hpw && task < Hq + Hkv) {
      const bool is_q = task < Hq;
      const __nv_bfloat16 *nw = is_q ? q_norm_w : k_norm_w;
      L::load(is_q ? q_in + b * q_stride + (size_t)task * D + e0
                   : k_new + b * kv_stride + (size_t)(task - Hq) * D + e0,
              x[k]);
      if (nw != nullptr) L::load(nw + e0, w[k]);
    }
  }
  const int p = pos[b];
  if (p < 0 || p >= T_cap) {
    if (threadIdx.x == 0 && task_block == 0 && error_word != nullptr)
      atomicOr(error_word, kErrPosSkipped);
    return;
  }
  for (int i = threadIdx.x; i < D / 2; i += kThreads) {
    float sn, cs;
    rope_sincos_turns(p, turns.v[i], sn, cs);
    s_cos[i] = cs;
    s_sin[i] = sn;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kMaxHeadsPerWarp; ++k) {
    const int task = (task_block * hpw + k) * kWarps + warp;
    if (k < hpw && task < Hq + Hkv)
      rotate_head_loaded<D>(x[k], w[k], task < Hq ? q_norm_w : k_norm_w, q_out, v_new, k_cache,
                            v_cache, Hq, Hkv, T_cap, kv_stride, inv, interleaved, eps, b, task,
                            p, s_cos, s_sin);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) qknorm_rope_append_kernel(
    const __nv_bfloat16 *q_in, __nv_bfloat16 *q_out, const __nv_bfloat16 *__restrict__ k_new,
    const __nv_bfloat16 *__restrict__ v_new, const __nv_bfloat16 *__restrict__ q_norm_w,
    const __nv_bfloat16 *__restrict__ k_norm_w, __nv_bfloat16 *__restrict__ k_cache,
    __nv_bfloat16 *__restrict__ v_cache, const int32_t *__restrict__ pos, int Hq, int Hkv,
    int T_cap, size_t q_stride, size_t kv_stride, const InvFreq inv, const RopeTurns turns,
    int interleaved, float eps, uint32_t *error_word, int hpw) {
  __shared__ float s_cos[D / 2];
  __shared__ float s_sin[D / 2];
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  qknorm_rope_block<D>(q_in, q_out, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, pos, Hq,
                       Hkv, T_cap, q_stride, kv_stride, inv, turns, interleaved, eps, error_word,
                       blockIdx.x, blockIdx.y, hpw, s_cos, s_sin);
}

// K1 and K2 of one decode step in a single launch: grid.y == 0 normalises row b of the
// hidden state, grid.y >= 1 rotates and appends heads of sequence b.
template <int D, int VPT>
__global__ void __launch_bounds__(kThreads) rms_rope_fused_kernel(
    const uint4 *__restrict__ x, uint4 *__restrict__ residual, const uint4 *__restrict__ nw_h,
    uint4 *__restrict__ y, int vec_per_row, float inv_hidden,
    __nv_bfloat16 *q, const __nv_bfloat16 *__restrict__ k_new,
    const __nv_bfloat16 *__restrict__ v_new, const __nv_bfloat16 *__restrict__ q_norm_w,
    const __nv_bfloat16 *__restrict__ k_norm_w, __nv_bfloat16 *__restrict__ k_cache,
    __nv_bfloat16 *__restrict__ v_cache, const int32_t *__restrict__ pos, int Hq, int Hkv,
    int T_cap, const InvFreq inv, const RopeTurns turns, int interleaved, float eps,
    uint32_t *error_word, int hpw) {
  __shared__ float s_cos[D / 2];
  __shared__ float s_sin[D / 2];
  __shared__ float warp_part[kThreads / 32];
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  if (blockIdx.y == 0)
    rmsnorm_row<VPT, kThreads>(x, residual, nw_h, y, blockIdx.x, vec_per_row, inv_hidden, eps,
                               warp_part);
  else
    qknorm_rope_block<D>(q, q, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, pos, Hq, Hkv,
                         T_cap, (size_t)Hq * D, (size_t)Hkv * D, inv, turns, interleaved, eps,
                         error_word, blockIdx.x, blockIdx.y - 1, hpw, s_cos, s_sin);
}

}  // namespace

InvFreq make_inv_freq(int D, double theta) {
  InvFreq inv;
  for (int i = 0; i < D / 2; ++i) inv.v[i] = pow(theta, -2.0 * (double)i / (double)D);
  return inv;
}

RopeTurns make_rope_turns(int D, const InvFreq &inv) {
  RopeTurns t{};
  const long double two_pi = 6.283185307179586476925286766559L;
  for (int i = 0; i < D / 2; ++i) {
    const long double f = (long double)inv.v[i] / two_pi;
    t.v[i] = (unsigned long long)llroundl(ldexpl(f, 64));  // f <= 1/(2 pi): below 2^62
  }
  return t;
}

cudaError_t launch_qknorm_rope_append_strided(const void *q_in, void *q_out, size_t q_stride,
                                              const void *k_new, const void *v_new,
                                              size_t kv_stride, const void *q_norm_w,
                                              const void *k_norm_w, void *k_cache, void *v_cache,
                                              const int32_t *pos, int B, int Hq, int Hkv, int D,
                                              int T_cap, const InvFreq &inv, int interleaved,
                                              float eps, uint32_t *error_word,
                                              cudaStream_t stream) {
  auto *qi = static_cast<const __nv_bfloat16 *>(q_in);
  auto *qp = static_cast<__nv_bfloat16 *>(q_out);
  auto *kn = static_cast<const __nv_bfloat16 *>(k_new);
  auto *vn = static_cast<const __nv_bfloat16 *>(v_new);
  auto *qw = static_cast<const __nv_bfloat16 *>(q_norm_w);
  auto *kw = static_cast<const __nv_bfloat16 *>(k_norm_w);
  auto *kc = static_cast<__nv_bfloat16 *>(k_cache);
  auto *vc = static_cast<__nv_bfloat16 *>(v_cache);
  const int hpw = heads_per_warp(B, Hq, Hkv);
  const dim3 grid(B, (Hq + Hkv + kWarps * hpw - 1) / (kWarps * hpw));
  const RopeTurns turns = make_rope_turns(D, inv);
  cudaError_t e;
  if (D == 128)
    e = launch_pdl(qknorm_rope_append_kernel<128>, grid, kThreads, 0, stream, qi, qp, kn, vn, qw,
                   kw, kc, vc, pos, Hq, Hkv, T_cap, q_stride, kv_stride, inv, turns, interleaved,
                   eps, error_word, hpw);
  else
    e = launch_pdl(qknorm_rope_append_kernel<64>, grid, kThreads, 0, stream, qi, qp, kn, vn, qw,
                   kw, kc, vc, pos, Hq, Hkv, T_cap, q_stride, kv_stride, inv, turns, interleaved,
                   eps, error_word, hpw);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_rms_rope_fused(const void *x, void *residual, const void *norm_w, void *y,
                                  int hidden, float eps, void *q, const void *k_new,
                                  const void *v_new, const void *q_norm_w, const void *k_norm_w,
                                  void *k_cache, void *v_cache, const int32_t *pos, int B, int Hq,
                                  int Hkv, int D, int T_cap, const InvFreq &inv, int interleaved,
                                  uint32_t *error_word, cudaStream_t stream) {
  const int vec = hidden / 8;
  const float inv_h = 1.0f / (float)hidden;
  auto *xp = static_cast<const uint4 *>(x);
  auto *rp = static_cast<uint4 *>(residual);
  auto *wp = static_cast<const uint4 *>(norm_w);
  auto *yp = static_cast<uint4 *>(y);
  auto *qp = static_cast<__nv_bfloat16 *>(q);
  auto *kn = static_cast<const __nv_bfloat16 *>(k_new);
  auto *vn = static_cast<const __nv_bfloat16 *>(v_new);
  auto *qw = static_cast<const __nv_bfloat16 *>(q_norm_w);
  auto *kw = static_cast<const __nv_bfloat16 *>(k_norm_w);
  auto *kc = static_cast<__nv_bfloat16 *>(k_cache);
  auto *vc = static_cast<__nv_bfloat16 *>(v_cache);
  const int hpw = heads_per_warp(B, Hq, Hkv);
  const dim3 grid(B, 1 + (Hq + Hkv + kWarps * hpw - 1) / (kWarps * hpw));
  const int vpt = (vec + kThreads - 1) / kThreads;
  const RopeTurns turns = make_rope_turns(D, inv);
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, grid, kThreads, 0, stream, xp, rp, wp, yp, vec, inv_h, qp, kn, vn,
                      qw, kw, kc, vc, pos, Hq, Hkv, T_cap, inv, turns, interleaved, eps,
                      error_word, hpw);
  };
  cudaError_t e;
  if (D == 128)
    e = vpt <= 1 ? go(rms_rope_fused_kernel<128, 1>) : vpt <= 2 ? go(rms_rope_fused_kernel<128, 2>)
        : vpt <= 4 ? go(rms_rope_fused_kernel<128, 4>) : go(rms_rope_fused_kernel<128, 8>);
  else
    e = vpt <= 1 ? go(rms_rope_fused_kernel<64, 1>) : vpt <= 2 ? go(rms_rope_fused_kernel<64, 2>)
        : vpt <= 4 ? go(rms_rope_fused_kernel<64, 4>) : go(rms_rope_fused_kernel<64, 8>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace decattn
