// One head of the rotation step of the decode step, done by one warp: the per-head
// QK-RMSNorm and RoPE of a query head (rotated in place or into q_out) or of a new key
// (rotated into its cache slot, with the value copied beside it). Shared by the rotation
// kernel and the fused RMSNorm + rotation kernel, so both form the same bits.
//
// cutileGPT README, "The current runtime includes" (fused QK-Norm + RoPE + KV-cache
// writes); fusedtok README, "Operators" (RoPE, interleaved and NeoX layouts, kv-cache
// pos_offset).
#pragma once

#include "dec_device.cuh"
#include "rope_angles.cuh"

namespace decattn {

// A head of D bf16 values spread over a warp: E consecutive values per lane.
template <int D>
struct Lanes;
template <>
struct Lanes<128> {
  static constexpr int kE = 4;
  __device__ static void load(const __nv_bfloat16 *p, float (&x)[4]) {
    uint2 v = *reinterpret_cast<const uint2 *>(p);
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  }
  __device__ static void store(__nv_bfloat16 *p, const float (&x)[4]) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  }
  __device__ static void copy(__nv_bfloat16 *dst, const __nv_bfloat16 *src) {
    *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(src);
  }
};
template <>
struct Lanes<64> {
  static constexpr int kE = 2;
  __device__ static void load(const __nv_bfloat16 *p, float (&x)[2]) {
    uint32_t v = *reinterpret_cast<const uint32_t *>(p);
    x[0] = bf16_lo(v); x[1] = bf16_hi(v);
  }
  __device__ static void store(__nv_bfloat16 *p, const float (&x)[2]) {
    *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(x[0], x[1]);
  }
  __device__ static void copy(__nv_bfloat16 *dst, const __nv_bfloat16 *src) {
    *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(src);
  }
};

// The cos and sin of the angles a lane's E elements turn by: NeoX element j < D/2 pairs
// with j + D/2 (16 lanes away), so lane l's element e uses angle (l mod 16) * E + e;
// interleaved elements 2i and 2i + 1 share angle i in the same lane.
template <int D>
struct LaneAngles {
  float c[Lanes<D>::kE], s[Lanes<D>::kE];
  __device__ static int index(int lane, int e, int interleaved) {
    return interleaved ? (lane * Lanes<D>::kE + e) >> 1 : (lane & 15) * Lanes<D>::kE + e;
  }
  // from a table of the sequence's D/2 angles
  __device__ void from_table(const float *s_cos, const float *s_sin, int interleaved) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int e = 0; e < Lanes<D>::kE; ++e) {
      const int i = index(lane, e, interleaved);
      c[e] = s_cos[i];
      s[e] = s_sin[i];
    }
  }
};

// The frequencies of a lane's E elements (inv_freq of each element's angle).
template <int D>
__device__ __forceinline__ void lane_freqs(const InvFreq &inv, int interleaved,
                                           double (&fr)[Lanes<D>::kE]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < Lanes<D>::kE; ++e) fr[e] = inv.v[LaneAngles<D>::index(lane, e, interleaved)];
}

// The rotation of one head held by a warp (x, and the norm weights w when has_norm):
// optional RMSNorm over D, then RoPE at position p into y. A key (is_k) keeps the stored
// copy within one bf16 ulp where the fp32 rotation cancels (rope_exact).
template <int D>
__device__ __forceinline__ void rotate_values(const float (&x_in)[Lanes<D>::kE],
                                              const float (&w)[Lanes<D>::kE], bool has_norm,
                                              bool is_k, const LaneAngles<D> &ang, int p,
                                              const double (&fr)[Lanes<D>::kE], int interleaved,
                                              float eps, float (&y)[Lanes<D>::kE]) {
  constexpr int E = Lanes<D>::kE;
  const int lane = threadIdx.x & 31;
  const float inv_d = 1.0f / (float)D;
  float x[E], xw[E];  // xw: exact pre-rotation values: raw, or raw times the norm weight
  float rstd = 1.f;
  if (has_norm) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(x_in[e], x_in[e], ss);
    ss = warp_sum(ss);
    rstd = rsqrtf(ss * inv_d + eps);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      xw[e] = x_in[e] * w[e];
      x[e] = x_in[e] * rstd * w[e];
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) xw[e] = x[e] = x_in[e];
  }
  if (!interleaved) {
    // NeoX: element j < D/2 pairs with j + D/2, which lives 16 lanes away.
    const bool first = lane < 16;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
      const float other_w = __shfl_xor_sync(0xffffffffu, xw[e], 16);
      const float c = ang.c[e], sn = ang.s[e];
      y[e] = first ? (x[e] * c - other * sn) : (other * sn + x[e] * c);
      if (is_k && rope_cancels(y[e], x[e], other))  // K: the stored copy within one ulp
        y[e] = rope_exact(p, fr[e], xw[e], other_w, rstd, !first);
    }
  } else {
    // Interleaved: element 2i pairs with 2i + 1, both in this lane.
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float c = ang.c[e], sn = ang.s[e];
      y[e] = x[e] * c - x[e + 1] * sn;
      y[e + 1] = x[e] * sn + x[e + 1] * c;
      if (is_k && rope_cancels(y[e], x[e], x[e + 1]))
        y[e] = rope_exact(p, fr[e], xw[e], xw[e + 1], rstd, false);
      if (is_k && rope_cancels(y[e + 1], x[e], x[e + 1]))
        y[e + 1] = rope_exact(p, fr[e], xw[e + 1], xw[e], rstd, true);
    }
  }
}

// One warp's part of the rotation step for sequence b at position p, with the head
// already loaded (x, and the norm weights w when nw is set): task < Hq is q head `task`
// (rotated into q_out), else KV head g = task - Hq (K rotated into cache slot p, V
// copied there). s_cos / s_sin hold the sequence's D/2 angles.
template <int D>
__device__ __forceinline__ void rotate_head_loaded(
    float (&x)[Lanes<D>::kE], const float (&w)[Lanes<D>::kE], const __nv_bfloat16 *nw,
    __nv_bfloat16 *q_out, const __nv_bfloat16 *__restrict__ v_new,
    __nv_bfloat16 *__restrict__ k_cache, __nv_bfloat16 *__restrict__ v_cache, int Hq, int Hkv,
    int T_cap, size_t kv_stride, const InvFreq &inv, int interleaved, float eps, int b,
    int task, int p, const float *s_cos, const float *s_sin) {
  using L = Lanes<D>;
  constexpr int E = L::kE;
  const int e0 = (threadIdx.x & 31) * E;  // first element of this lane
  const bool is_q = task < Hq;
  const int g = task - Hq;
  LaneAngles<D> ang;
  ang.from_table(s_cos, s_sin, interleaved);
  double fr[E] = {};
  if (!is_q) lane_freqs<D>(inv, interleaved, fr);  // for the exact path of a cancelling K
  float y[E];
  rotate_values<D>(x, w, nw != nullptr, !is_q, ang, p, fr, interleaved, eps, y);
  if (is_q) {
    L::store(q_out + ((size_t)b * Hq + task) * D + e0, y);
  } else {
    const size_t slot = (((size_t)b * Hkv + g) * T_cap + p) * D + e0;
    L::store(k_cache + slot, y);
    L::copy(v_cache + slot, v_new + b * kv_stride + (size_t)g * D + e0);
  }
}

}  // namespace decattn
