// K1: RMSNorm with a fused residual add, one CTA per row.
//
// fusedtok README, "Operators" (RMSNorm (+residual), fused residual add) and
// "Usage" (h = rmsnorm(h, w, residual=h)); cutileGPT README, "Why tiles"
// (rstd = 1/sqrt(sum(x*x)/N + eps), y = x * rstd * w).
//
// The row body lives in rmsnorm_body.cuh (shared with the fused K1+K2 launch).
#include "dec_launch.h"
#include "rmsnorm_body.cuh"

namespace decattn {
namespace {

constexpr int kThreads = 256;

template <int VPT>
__global__ void __launch_bounds__(kThreads) rmsnorm_residual_kernel(
    const uint4 *__restrict__ x, uint4 *__restrict__ residual, const uint4 *__restrict__ w,
    uint4 *__restrict__ y, int vec_per_row, float inv_hidden, float eps) {
  __shared__ float warp_part[kThreads / 32];
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  rmsnorm_row<VPT, kThreads>(x, residual, w, y, blockIdx.x, vec_per_row, inv_hidden, eps,
                             warp_part);
}

}  // namespace

cudaError_t launch_rmsnorm_residual(const void *x, void *residual, const void *weight, void *y,
                                    int B, int hidden, float eps, cudaStream_t stream) {
  const int vec = hidden / 8;
  const int vpt = (vec + kThreads - 1) / kThreads;
  const float inv_h = 1.0f / (float)hidden;
  const uint4 *xp = static_cast<const uint4 *>(x);
  uint4 *rp = static_cast<uint4 *>(residual);
  const uint4 *wp = static_cast<const uint4 *>(weight);
  uint4 *yp = static_cast<uint4 *>(y);
  cudaError_t e;
  if (vpt <= 1)
    e = launch_pdl(rmsnorm_residual_kernel<1>, B, kThreads, 0, stream, xp, rp, wp, yp, vec, inv_h, eps);
  else if (vpt <= 2)
    e = launch_pdl(rmsnorm_residual_kernel<2>, B, kThreads, 0, stream, xp, rp, wp, yp, vec, inv_h, eps);
  else if (vpt <= 4)
    e = launch_pdl(rmsnorm_residual_kernel<4>, B, kThreads, 0, stream, xp, rp, wp, yp, vec, inv_h, eps);
  else
    e = launch_pdl(rmsnorm_residual_kernel<8>, B, kThreads, 0, stream, xp, rp, wp, yp, vec, inv_h, eps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace decattn
