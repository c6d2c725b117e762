// Device body of K1 (RMSNorm with a fused residual add) for one row, shared by the
// standalone kernel and the fused K1+K2 launch of the decode step.
//
// fusedtok README, "Operators" (RMSNorm (+residual), fused residual add) and
// "Usage" (h = rmsnorm(h, w, residual=h)); cutileGPT README, "Why tiles"
// (rstd = 1/sqrt(sum(x*x)/N + eps), y = x * rstd * w).
#pragma once

#include "dec_device.cuh"

namespace decattn {

// Each thread owns up to VPT 16-byte vectors (8 bf16) of the row, keeps the fp32 sum
// s = x + residual in registers, writes bf16(s) back as the new residual, and after
// one block reduction of sum(s^2) writes y = bf16(s * rstd * w). The row is read
// once and written once. `warp_part` is THREADS/32 floats of shared memory.
template <int VPT, int THREADS>
__device__ __forceinline__ void rmsnorm_row(const uint4 *__restrict__ x, uint4 *__restrict__ residual,
                                            const uint4 *__restrict__ w, uint4 *__restrict__ y,
                                            int row, int vec_per_row, float inv_hidden, float eps,
                                            float *warp_part) {
  const long long row_off = (long long)row * vec_per_row;
  float s[VPT][8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * THREADS;
    if (v < vec_per_row) {
      uint4 xv = __ldg(x + row_off + v);
      uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t rw[4] = {0u, 0u, 0u, 0u};
      if (residual != nullptr) {
        uint4 rv = residual[row_off + v];
        rw[0] = rv.x; rw[1] = rv.y; rw[2] = rv.z; rw[3] = rv.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        s[j][2 * k] = bf16_lo(xw[k]) + bf16_lo(rw[k]);
        s[j][2 * k + 1] = bf16_hi(xw[k]) + bf16_hi(rw[k]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(s[j][k], s[j][k], ss);
      if (residual != nullptr) {
        uint4 o;
        o.x = pack_bf16x2(s[j][0], s[j][1]);
        o.y = pack_bf16x2(s[j][2], s[j][3]);
        o.z = pack_bf16x2(s[j][4], s[j][5]);
        o.w = pack_bf16x2(s[j][6], s[j][7]);
        residual[row_off + v] = o;
      }
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < THREADS / 32; ++i) tot += warp_part[i];
  const float rstd = rsqrtf(tot * inv_hidden + eps);
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * THREADS;
    if (v < vec_per_row) {
      uint4 wv = __ldg(w + v);
      uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        o[k] = pack_bf16x2(s[j][2 * k] * rstd * bf16_lo(ww[k]),
                           s[j][2 * k + 1] * rstd * bf16_hi(ww[k]));
      y[row_off + v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace decattn
