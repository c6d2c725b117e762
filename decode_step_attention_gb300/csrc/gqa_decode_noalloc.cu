// dec_gqa_decode_attn_noalloc: decode attention for callers that cannot allocate.
//
// The regular attention call needs a caller-provided workspace for the split
// partials. Some callers have no way to get one: code that runs inside a host
// callback or a custom allocator hook (where calling cudaMalloc would re-enter the
// allocator or deadlock), plugins embedded in a runtime that owns every device
// allocation and hands out none, or tools that must not change the process's
// memory footprint after start-up. For them this file keeps one fixed scratch
// buffer in static device memory, and the entry point below runs the usual split
// pass and merge with it. Nothing here calls cudaMalloc, cudaFree or any library
// routine that allocates.
//
// The scratch buffer is a file-scope __device__ array of kNoAllocScratchBytes
// (4 MiB). Every GPU that loads this library holds it until the process exits.
// All calls on a device share it: two calls whose kernels overlap on the GPU (on
// different streams, say) race on it and produce garbage, so serialise them.
// The buffer keeps whatever the previous call left; the part that must start at
// zero, the header with the device error word and the split pass's claim counters,
// is cleared by each call on its stream before the kernels run.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the first call on each device looks the address
// up with cudaGetSymbolAddress while that device is current and caches it. That
// first call may also load the module on the device, so make it before any stream
// capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "decattn.h"
#include "dec_launch.h"

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
dec_status scratch_address(int device, void **addr) {
  if (device < 0 || device >= kMaxDevices)
    return decattn::record_error(DEC_ERR_UNSUPPORTED, "device ordinal beyond the scratch table");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[device] == nullptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return decattn::record_error(DEC_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_scratch_addr[device] = p;
  }
  *addr = g_scratch_addr[device];
  return DEC_OK;
}

}  // namespace

extern "C" dec_status dec_gqa_decode_attn_noalloc(const void *q, const void *k_cache,
                                                  const void *v_cache, const int32_t *lens,
                                                  void *out, int B, int Hq, int Hkv, int D,
                                                  int T_cap, int max_len, float scale,
                                                  int num_parts, dec_stream_t stream) {
  if (B == 0) return dec_gqa_decode_attn(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap,
                                         max_len, scale, num_parts, nullptr, 0, stream);
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_parts < 0)
    return decattn::record_error(DEC_ERR_INVALID_ARG, "bad batch, head counts or num_parts");
  const size_t need = dec_attn_workspace_bytes(B, Hq, Hkv, D, max_len, num_parts);
  if (need > kNoAllocScratchBytes)
    return decattn::record_error(DEC_ERR_WORKSPACE,
                                 "this shape needs more scratch than the 4 MiB static buffer; "
                                 "use dec_gqa_decode_attn with a workspace");
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess)
    return decattn::record_error(DEC_ERR_CUDA, "cudaGetDevice failed");
  void *scratch = nullptr;
  dec_status st = scratch_address(device, &scratch);
  if (st != DEC_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 4 * sizeof(uint32_t), s) != cudaSuccess)
    return decattn::record_error(DEC_ERR_CUDA, "clearing the scratch header failed");
  return dec_gqa_decode_attn(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale,
                             num_parts, scratch, kNoAllocScratchBytes, stream);
}
