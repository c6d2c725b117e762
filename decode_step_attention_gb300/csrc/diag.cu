// dec_diag_wait_timeout: exercises the bounded pipeline wait the kernels use.
//
// A one-warp kernel waits on a shared-memory mbarrier that nothing ever arrives at,
// using the same bounded wait as the split pass; when the wait gives up it raises
// DEC_DEVERR_WAIT_TIMEOUT in the caller's error word and returns, so the context
// stays usable. This is how a stalled pipeline shows up to the host.
#include "dec_device.cuh"
#include "dec_launch.h"

namespace decattn {
namespace {

__global__ void wait_timeout_kernel(uint32_t *error_word) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const bool done = mbar_wait_bounded(b, 0);  // phase 0 never completes
  __syncwarp();
  if (!done && threadIdx.x == 0) atomicOr(error_word, kErrWaitTimeout);
}

}  // namespace
}  // namespace decattn

extern "C" dec_status dec_diag_wait_timeout(uint32_t *error_word, dec_stream_t stream) {
  if (error_word == nullptr || (reinterpret_cast<uintptr_t>(error_word) & 3u) != 0)
    return decattn::record_error(DEC_ERR_INVALID_ARG, "error_word must be a 4-byte aligned device pointer");
  decattn::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(error_word);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return decattn::record_error(DEC_ERR_CUDA, cudaGetErrorString(e));
  return DEC_OK;
}
