// K1: RMSNorm with a fused residual add, one CTA per row.
//
// fusedtok README, "Operators" (RMSNorm (+residual), fused residual add) and
// "Usage" (h = rmsnorm(h, w, residual=h)); cutileGPT README, "Why tiles"
// (rstd = 1/sqrt(sum(x*x)/N + eps), y = x * rstd * w).
//
// The row body lives in rmsnorm_body.cuh (shared with the fused K1+K2 launch).
#include <atomic>

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

// K1 often runs on a second stream beside the split pass, whose single CTA per SM
// takes nearly all of the SM's shared memory. An SM runs blocks of different kernels
// side by side only under one shared-memory carveout, so K1 asks for the largest
// carveout too: its blocks then fit next to a split CTA instead of waiting for the
// SM to drain. (It needs no L1 capacity: every byte it touches is read once.)
template <int VPT>
cudaError_t prefer_max_shared() {
  static std::atomic<unsigned long long> done{0};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (device & 63);
  if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(rmsnorm_residual_kernel<VPT>,
                           cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

template <int VPT>
cudaError_t launch_vpt(int B, cudaStream_t stream, const uint4 *xp, uint4 *rp, const uint4 *wp,
                       uint4 *yp, int vec, float inv_h, float eps) {
  const cudaError_t e = prefer_max_shared<VPT>();
  if (e != cudaSuccess) return e;
  return launch_pdl(rmsnorm_residual_kernel<VPT>, B, kThreads, 0, stream, xp, rp, wp, yp, vec,
                    inv_h, eps);
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
    e = launch_vpt<1>(B, stream, xp, rp, wp, yp, vec, inv_h, eps);
  else if (vpt <= 2)
    e = launch_vpt<2>(B, stream, xp, rp, wp, yp, vec, inv_h, eps);
  else if (vpt <= 4)
    e = launch_vpt<4>(B, stream, xp, rp, wp, yp, vec, inv_h, eps);
  else
    e = launch_vpt<8>(B, stream, xp, rp, wp, yp, vec, inv_h, eps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace decattn
