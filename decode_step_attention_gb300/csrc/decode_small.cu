// The whole decode step in one launch, for problems too small to fill the GPU: K1
// (RMSNorm with the residual add), K2 (QK-norm, RoPE, K/V append) and the attention
// with its merge, where three launches' latencies would otherwise dominate.
//
// fusedtok README, "Operators" (RMSNorm (+residual); RoPE in NeoX and interleaved
// layouts with a kv-cache position offset; attention_decode with online softmax, a
// flash-decoding split and per-sequence lengths) and "Usage"; cutileGPT README, "The
// current runtime includes" (fused QK-Norm + RoPE + KV-cache writes, fewer launches).
//
// Grid (S, Hkv + 1, B), clusters of S CTAs along x. Cluster (g, b), g < Hkv, serves KV
// head g of sequence b: every CTA forms the group's rotated query heads and the new
// token's K from the raw inputs (rounded to bf16 as the stored copies are), streams an
// S-th of the sequence's rows (the new row from its own copy, the others from the
// cache), and pushes its softmax state into CTA 0's shared memory (distributed shared
// memory stores); after one cluster barrier CTA 0 merges them, writes the output heads,
// and only then the rotated queries in place (every CTA of the cluster has read the raw
// ones by that barrier); it also writes the new K/V slot, which no CTA reads from the
// cache. Cluster g == Hkv: its CTA 0 normalises row
// b of the hidden state. Arithmetic as in the standalone kernels: fp32, angles from
// fp64 inv_freq, scores in base 2 (q prescaled by scale * log2 e).
//
// Without positions (pos == nullptr) the same kernel is the attention call alone for
// short contexts: q is taken as already rotated and the cache as already appended, no
// RMSNorm cluster is launched, and nothing but the output is written — the split pass
// and its merge in one launch.
#include <math.h>

#include "dec_device.cuh"
#include "dec_launch.h"
#include "rmsnorm_body.cuh"
#include "rope_angles.cuh"

namespace decattn {
namespace {

constexpr int kSmThreads = 256;
constexpr int kSmWarps = kSmThreads / 32;
constexpr int kSmMaxG = 8;       // query heads per KV head
constexpr int kSmRowBatch = 8;   // rows a warp loads before it uses them
constexpr int kSmTogether = 2;   // rows whose scores are reduced and applied together
constexpr int kSmMaxSplit = 8;   // CTAs per (sequence, KV head): a portable cluster

struct SmallArgs {
  const uint4 *x;
  uint4 *residual;
  const uint4 *norm_w;
  uint4 *y;
  int vec_per_row;
  float inv_hidden, eps;
  __nv_bfloat16 *q;
  const __nv_bfloat16 *k_new, *v_new, *q_norm_w, *k_norm_w;
  __nv_bfloat16 *k_cache, *v_cache;
  const int32_t *pos, *lens;
  __nv_bfloat16 *out;
  int Hq, Hkv, T_cap, interleaved, window;
  float scale_log2;
  uint32_t *error_word;
  InvFreq inv;      // fp64 frequencies (the exact path of a cancelling K)
  RopeTurns turns;  // the same as fractions of a turn (the angles)
};

template <int D>
struct Row;
template <>
struct Row<128> {
  using T = uint2;
  static constexpr int kE = 4;
  __device__ static void unpack(T v, float (&x)[4]) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  }
  __device__ static T pack(const float (&x)[4]) {
    return make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  }
};
template <>
struct Row<64> {
  using T = uint32_t;
  static constexpr int kE = 2;
  __device__ static void unpack(T v, float (&x)[2]) { x[0] = bf16_lo(v); x[1] = bf16_hi(v); }
  __device__ static T pack(const float (&x)[2]) { return pack_bf16x2(x[0], x[1]); }
};

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_peer_f32(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

template <int D, int VPT>
__global__ void __launch_bounds__(kSmThreads) decode_small_kernel(const SmallArgs a) {
  using R = Row<D>;
  constexpr int E = R::kE;
  constexpr int kStride = D + 4;  // floats per partial state: acc[D], m, l, 2 pad (16 B rows)
  __shared__ float s_cos[D / 2], s_sin[D / 2];
  __shared__ float s_q[kSmMaxG][D];  // rotated query heads (bf16 values), times scale log2 e
  __shared__ float s_k[D], s_v[D];   // the new token's K (rotated, bf16 values) and V
  __shared__ __align__(16) float s_warp[kSmWarps][kSmMaxG][kStride];
  __shared__ float warp_part[kSmWarps];
  // CTA 0: the states every CTA of the cluster pushes, [S][kSmMaxG][kStride] floats
  extern __shared__ __align__(16) float s_recv[];

  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int b = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- K1 (one CTA)
  if (g == a.Hkv) {
    if (blockIdx.x == 0)
      rmsnorm_row<VPT, kSmThreads>(a.x, a.residual, a.norm_w, a.y, b, a.vec_per_row,
                                   a.inv_hidden, a.eps, warp_part);
    return;  // this cluster uses no cluster barrier
  }

  const uint32_t S = gridDim.x, rank = cluster_rank_x();
  const int G = a.Hq / a.Hkv;
  const int e0 = lane * E;
  const bool attn_only = a.pos == nullptr;
  const int last_task = attn_only ? G - 1 : G;  // the K head's task is task G
  // Every input that depends on nothing else is requested first, so that their
  // latencies overlap: the position, the length, this warp's heads (G query heads,
  // then the new K, two tasks at most per warp), their norm weights and the new V.
  const int p = attn_only ? -1 : a.pos[b];
  int L = a.lens[b];
  typename R::T raw[2], wraw[2], vraw = {};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int task = warp + j * kSmWarps;
    if (task > last_task) break;
    const bool is_q = task < G;
    const __nv_bfloat16 *src = is_q ? a.q + ((size_t)b * a.Hq + (size_t)g * G + task) * D
                                    : a.k_new + ((size_t)b * a.Hkv + g) * D;
    raw[j] = *reinterpret_cast<const typename R::T *>(src + e0);
    const __nv_bfloat16 *nw = is_q ? a.q_norm_w : a.k_norm_w;
    if (nw != nullptr) wraw[j] = *reinterpret_cast<const typename R::T *>(nw + e0);
    if (!is_q)
      vraw = *reinterpret_cast<const typename R::T *>(a.v_new + ((size_t)b * a.Hkv + g) * D + e0);
  }
  const bool rotate = !attn_only && p >= 0 && p < a.T_cap;
  if (!attn_only && !rotate && rank == 0 && g == 0 && threadIdx.x == 0 &&
      a.error_word != nullptr)
    atomicOr(a.error_word, kErrPosSkipped);
  if (L < 0 || L > a.T_cap) {
    if (rank == 0 && g == 0 && threadIdx.x == 0 && a.error_word != nullptr)
      atomicOr(a.error_word, kErrLenClamped);
    L = L < 0 ? 0 : a.T_cap;
  }
  const int start = (a.window > 0 && L > a.window) ? L - a.window : 0;
  const int chunk = (L - start + (int)S - 1) / (int)S;
  const int r0 = start + (int)rank * chunk;
  const int r1 = min(L, r0 + chunk);
  // this warp's first batch of cache rows, in flight while the rotation is formed
  const __nv_bfloat16 *kbase = a.k_cache + ((size_t)b * a.Hkv + g) * a.T_cap * D + e0;
  const __nv_bfloat16 *vbase = a.v_cache + ((size_t)b * a.Hkv + g) * a.T_cap * D + e0;
  typename R::T kr[kSmRowBatch] = {}, vr[kSmRowBatch] = {};
  auto load_batch = [&](int base) {
#pragma unroll
    for (int i = 0; i < kSmRowBatch; ++i) {  // every load of the batch in flight at once
      const int t = base + i * kSmWarps;
      if (t < r1 && !(rotate && t == p)) {
        kr[i] = *reinterpret_cast<const typename R::T *>(kbase + (size_t)t * D);
        vr[i] = *reinterpret_cast<const typename R::T *>(vbase + (size_t)t * D);
      }
    }
  };
  load_batch(r0 + warp);

  // --------------------------------------------------------------------- K2
  if (rotate)
    for (int i = threadIdx.x; i < D / 2; i += kSmThreads) {
      float sn, cs;
      rope_sincos_turns(p, a.turns.v[i], sn, cs);
      s_cos[i] = cs;
      s_sin[i] = sn;
    }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 2; ++j) {  // G query heads, then the K head
    const int task = warp + j * kSmWarps;
    if (task > last_task) break;
    const bool is_q = task < G;
    float x[E];
    R::unpack(raw[j], x);
    if (rotate) {
      float xw[E];  // exact pre-rotation values: raw, or raw times the norm weight
      float rstd = 1.f;
      if ((is_q ? a.q_norm_w : a.k_norm_w) != nullptr) {
        float w[E];
        R::unpack(wraw[j], w);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
        ss = warp_sum(ss);
        rstd = rsqrtf(ss * (1.0f / (float)D) + a.eps);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          xw[e] = x[e] * w[e];
          x[e] = x[e] * rstd * w[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) xw[e] = x[e];
      }
      float yv[E];
      if (!a.interleaved) {
        // NeoX: element j < D/2 pairs with j + D/2, which lives 16 lanes away
        const bool first = lane < 16;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
          const float other_w = __shfl_xor_sync(0xffffffffu, xw[e], 16);
          const int i = (lane & 15) * E + e;
          yv[e] = first ? (x[e] * s_cos[i] - other * s_sin[i])
                        : (other * s_sin[i] + x[e] * s_cos[i]);
          // K: a cancelling element again in fp64 (as the rotation call does)
          if (!is_q && rope_cancels(yv[e], x[e], other))
            yv[e] = rope_exact(p, a.inv.v[i], xw[e], other_w, rstd, !first);
        }
      } else {
        // interleaved: element 2i pairs with 2i + 1, both in this lane
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const int i = (e0 + e) >> 1;
          yv[e] = x[e] * s_cos[i] - x[e + 1] * s_sin[i];
          yv[e + 1] = x[e] * s_sin[i] + x[e + 1] * s_cos[i];
          if (!is_q && rope_cancels(yv[e], x[e], x[e + 1]))
            yv[e] = rope_exact(p, a.inv.v[i], xw[e], xw[e + 1], rstd, false);
          if (!is_q && rope_cancels(yv[e + 1], x[e], x[e + 1]))
            yv[e + 1] = rope_exact(p, a.inv.v[i], xw[e + 1], xw[e], rstd, true);
        }
      }
      // the stored copies are bf16: use exactly those values
      R::unpack(R::pack(yv), x);
    }
    if (is_q) {
#pragma unroll
      for (int e = 0; e < E; ++e) s_q[task][e0 + e] = x[e] * a.scale_log2;
    } else {
      float v[E];
      R::unpack(vraw, v);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        s_k[e0 + e] = x[e];
        s_v[e0 + e] = v[e];
      }
    }
  }
  __syncthreads();

  // --------------------------------------------------------------- attention
  float qv[kSmMaxG][E], acc[kSmMaxG][E], m[kSmMaxG], l[kSmMaxG];
#pragma unroll
  for (int h = 0; h < kSmMaxG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qv[h][e] = h < G ? s_q[h][e0 + e] : 0.f;
      acc[h][e] = 0.f;
    }
  }
  for (int base = r0 + warp; base < r1; base += kSmWarps * kSmRowBatch) {
    if (base != r0 + warp) load_batch(base);  // the first batch is already in flight
    // kSmTogether rows at a time: their reductions are independent shuffle chains that
    // overlap, and one rescale of the running state serves all of them
#pragma unroll
    for (int i = 0; i < kSmRowBatch; i += kSmTogether) {
      if (base + i * kSmWarps >= r1) break;
      float kk[kSmTogether][E], vv[kSmTogether][E];
      bool live[kSmTogether];
#pragma unroll
      for (int j = 0; j < kSmTogether; ++j) {
        const int t = base + (i + j) * kSmWarps;
        live[j] = t < r1;
        if (rotate && t == p) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            kk[j][e] = s_k[e0 + e];
            vv[j][e] = s_v[e0 + e];
          }
        } else {
          R::unpack(kr[i + j], kk[j]);  // unused when the row is past r1
          R::unpack(vr[i + j], vv[j]);
        }
      }
#pragma unroll
      for (int h = 0; h < kSmMaxG; ++h) {
        if (h >= G) break;
        float d[kSmTogether];
#pragma unroll
        for (int j = 0; j < kSmTogether; ++j) {
          d[j] = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) d[j] = fmaf(qv[h][e], kk[j][e], d[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int j = 0; j < kSmTogether; ++j) d[j] += __shfl_xor_sync(0xffffffffu, d[j], o);
        float mn = m[h];
#pragma unroll
        for (int j = 0; j < kSmTogether; ++j) {
          if (!live[j]) d[j] = -INFINITY;  // rows past r1 add nothing
          mn = fmaxf(mn, d[j]);
        }
        const float c = exp2f(m[h] - mn);
        float pj[kSmTogether], psum = 0.f;
#pragma unroll
        for (int j = 0; j < kSmTogether; ++j) {
          pj[j] = exp2f(d[j] - mn);
          psum += pj[j];
        }
        l[h] = fmaf(l[h], c, psum);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          float add = 0.f;
#pragma unroll
          for (int j = 0; j < kSmTogether; ++j) add = fmaf(pj[j], vv[j][e], add);
          acc[h][e] = fmaf(acc[h][e], c, add);
        }
        m[h] = mn;
      }
    }
  }
  // this warp's states, then the CTA's: warp h combines head h over the warps
#pragma unroll
  for (int h = 0; h < kSmMaxG; ++h) {
    if (h >= G) break;
#pragma unroll
    for (int e = 0; e < E; ++e) s_warp[warp][h][e0 + e] = acc[h][e];
    if (lane == 0) {
      s_warp[warp][h][D] = m[h];
      s_warp[warp][h][D + 1] = l[h];
    }
  }
  __syncthreads();
  if (warp < G) {
    const int h = warp;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSmWarps; ++w) M = fmaxf(M, s_warp[w][h][D]);
    float tot = 0.f, r[E];
#pragma unroll
    for (int e = 0; e < E; ++e) r[e] = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kSmWarps; ++w) {
        const float mw = s_warp[w][h][D];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        tot = fmaf(f, s_warp[w][h][D + 1], tot);
#pragma unroll
        for (int e = 0; e < E; ++e) r[e] = fmaf(f, s_warp[w][h][e0 + e], r[e]);
      }
    }
    // push this CTA's state of head h into CTA 0's shared memory
    float *slot = s_recv + ((size_t)rank * kSmMaxG + h) * kStride;
#pragma unroll
    for (int e = 0; e < E; ++e) st_peer_f32(peer_addr(slot + e0 + e, 0), r[e]);
    if (lane == 0) {
      st_peer_f32(peer_addr(slot + D, 0), M);
      st_peer_f32(peer_addr(slot + D + 1, 0), tot);
    }
  }
  // every state is in CTA 0 and every raw q has been read; the other CTAs may leave,
  // since CTA 0 reads only its own shared memory from here on
  cluster_barrier();

  // ------------------------------------ merge (CTA 0), append, rotated q in place
  // The append comes after the barrier: no CTA reads the slot from the cache, and
  // stores issued before it would hold up the barrier's release.
  if (rank == 0 && rotate && warp == kSmWarps - 1) {
    float kk[E], vv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kk[e] = s_k[e0 + e];
      vv[e] = s_v[e0 + e];
    }
    const size_t slot = (((size_t)b * a.Hkv + g) * a.T_cap + p) * D + e0;
    *reinterpret_cast<typename R::T *>(a.k_cache + slot) = R::pack(kk);
    *reinterpret_cast<typename R::T *>(a.v_cache + slot) = R::pack(vv);
  }
  if (rank == 0 && warp < G) {
    const int h = warp;
    float pm[kSmMaxSplit], pl[kSmMaxSplit], pa[kSmMaxSplit][E];
#pragma unroll
    for (uint32_t c = 0; c < kSmMaxSplit; ++c)
      if (c < S) {
        const float *st = s_recv + ((size_t)c * kSmMaxG + h) * kStride;
        pm[c] = st[D];
        pl[c] = st[D + 1];
#pragma unroll
        for (int e = 0; e < E; ++e) pa[c][e] = st[e0 + e];
      }
    float M = -INFINITY;
#pragma unroll
    for (uint32_t c = 0; c < kSmMaxSplit; ++c)
      if (c < S) M = fmaxf(M, pm[c]);
    float tot = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (uint32_t c = 0; c < kSmMaxSplit; ++c)
        if (c < S && pm[c] > -INFINITY) {
          const float f = exp2f(pm[c] - M);
          tot = fmaf(f, pl[c], tot);
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = fmaf(f, pa[c][e], o[e]);
        }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;  // an empty sequence gives zeros
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= inv;
    const size_t head = ((size_t)b * a.Hq + (size_t)g * G + h) * D + e0;
    *reinterpret_cast<typename R::T *>(a.out + head) = R::pack(o);
    if (rotate) {
      float qq[E];
#pragma unroll
      for (int e = 0; e < E; ++e) qq[e] = s_q[h][e0 + e] / a.scale_log2;
      *reinterpret_cast<typename R::T *>(a.q + head) = R::pack(qq);
    }
  }
}

}  // namespace

namespace {
cudaError_t launch_small(const SmallArgs &a, int D, int hidden, int B, int splits,
                         bool with_norm, cudaStream_t stream);
}  // namespace

// CTAs per (sequence, KV head) for the one-launch step, 0 when the problem is too big
// for it (or of a shape it does not cover): short contexts, a few (sequence, head)
// pairs, at most 8 query heads per KV head.
int small_step_splits(int B, int Hq, int Hkv, int D, int max_len, int window) {
  if (B < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > kSmMaxG || (D != 64 && D != 128))
    return 0;
  const int rows = (window > 0 && window < max_len) ? window : max_len;
  if (rows > kSmallMaxRows || (long long)B * Hkv > kSmallMaxPairs) return 0;
  int s = (rows + 15) / 16;  // about 2 rows per warp before the split reaches 8
  return s < 1 ? 1 : (s > kSmMaxSplit ? kSmMaxSplit : s);
}

cudaError_t launch_decode_small(const void *x, void *residual, const void *norm_w, void *y,
                                int hidden, float eps, void *q, const void *k_new,
                                const void *v_new, const void *q_norm_w, const void *k_norm_w,
                                void *k_cache, void *v_cache, const int32_t *pos,
                                const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                                int T_cap, int splits, int window, float scale_log2,
                                const InvFreq &inv, int interleaved, uint32_t *error_word,
                                cudaStream_t stream) {
  SmallArgs a{};
  a.x = static_cast<const uint4 *>(x);
  a.residual = static_cast<uint4 *>(residual);
  a.norm_w = static_cast<const uint4 *>(norm_w);
  a.y = static_cast<uint4 *>(y);
  a.vec_per_row = hidden / 8;
  a.inv_hidden = 1.0f / (float)hidden;
  a.eps = eps;
  a.q = static_cast<__nv_bfloat16 *>(q);
  a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  a.q_norm_w = static_cast<const __nv_bfloat16 *>(q_norm_w);
  a.k_norm_w = static_cast<const __nv_bfloat16 *>(k_norm_w);
  a.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
  a.pos = pos;
  a.lens = lens;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.T_cap = T_cap;
  a.interleaved = interleaved;
  a.window = window;
  a.scale_log2 = scale_log2;
  a.error_word = error_word;
  a.inv = inv;
  a.turns = make_rope_turns(D, inv);
  return launch_small(a, D, hidden, B, splits, true, stream);
}

cudaError_t launch_attn_small(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                              int T_cap, int splits, int window, float scale_log2,
                              uint32_t *error_word, cudaStream_t stream) {
  SmallArgs a{};
  a.q = static_cast<__nv_bfloat16 *>(const_cast<void *>(q));  // read only: no positions
  a.k_cache = static_cast<__nv_bfloat16 *>(const_cast<void *>(k_cache));
  a.v_cache = static_cast<__nv_bfloat16 *>(const_cast<void *>(v_cache));
  a.pos = nullptr;
  a.lens = lens;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.T_cap = T_cap;
  a.window = window;
  a.scale_log2 = scale_log2;
  a.error_word = error_word;
  return launch_small(a, D, 8, B, splits, false, stream);
}

namespace {
// Grid (splits, Hkv (+ 1 for the RMSNorm cluster), B), clusters of `splits` along x.
cudaError_t launch_small(const SmallArgs &a, int D, int hidden, int B, int splits,
                         bool with_norm, cudaStream_t stream) {
  if (splits < 1 || splits > kSmMaxSplit) return cudaErrorInvalidValue;
  const int Hkv = a.Hkv;
  const int vpt = (hidden / 8 + kSmThreads - 1) / kSmThreads;
  void (*kern)(const SmallArgs);
  if (D == 128)
    kern = vpt <= 1 ? decode_small_kernel<128, 1> : vpt <= 2 ? decode_small_kernel<128, 2>
         : vpt <= 4 ? decode_small_kernel<128, 4> : decode_small_kernel<128, 8>;
  else
    kern = vpt <= 1 ? decode_small_kernel<64, 1> : vpt <= 2 ? decode_small_kernel<64, 2>
         : vpt <= 4 ? decode_small_kernel<64, 4> : decode_small_kernel<64, 8>;
  const size_t recv = (size_t)splits * kSmMaxG * (D + 4) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)recv);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits, (unsigned)(Hkv + (with_norm ? 1 : 0)), (unsigned)B);
  cfg.blockDim = dim3(kSmThreads);
  cfg.dynamicSmemBytes = recv;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

}  // namespace decattn
