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
// zero (the device error word, the split pass's claim counters and the one-launch
// attention's counters, the first 28 bytes of the header) is cleared by each call on
// its stream before the kernels run, and only after every argument check has passed (a
// refused call enqueues nothing). The launch epoch after them is kept: it tells this
// call's piece marks from the ones earlier calls left in the buffer.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so every call looks the address up with
// cudaGetSymbolAddress on the current device. The lookup is cheap once the module
// is loaded, and doing it on every call keeps it right after the device's context
// has been reset or recreated (the array then lives at a new address). The first
// call on a device may load the module there, so make it before any stream capture.
#include <cuda_runtime.h>

#include "decattn.h"
#include "dec_launch.h"

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" dec_status dec_gqa_decode_attn_noalloc(const void *q, const void *k_cache,
                                                  const void *v_cache, const int32_t *lens,
                                                  void *out, int B, int Hq, int Hkv, int D,
                                                  int T_cap, int max_len, float scale,
                                                  int num_parts, uint32_t *error_word,
                                                  dec_stream_t stream) {
  if (B == 0) return dec_gqa_decode_attn(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap,
                                         max_len, scale, num_parts, nullptr, 0, stream);
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_parts < 0)
    return decattn::record_error(DEC_ERR_INVALID_ARG, "bad batch, head counts or num_parts");
  const size_t need = dec_attn_workspace_bytes(B, Hq, Hkv, D, max_len, num_parts);
  if (need == 0 || need > kNoAllocScratchBytes)
    return decattn::record_error(DEC_ERR_WORKSPACE,
                                 "this shape needs more scratch than the 4 MiB static buffer; "
                                 "use dec_gqa_decode_attn with a workspace");
  void *scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr) {
    (void)cudaGetLastError();
    return decattn::record_error(DEC_ERR_CUDA,
                                 "cudaGetSymbolAddress of the static scratch failed");
  }
  // every check of the attention call, then error_word's, before anything is enqueued
  dec_status st = decattn::attn_check(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap,
                                      max_len, scale, num_parts, scratch, kNoAllocScratchBytes);
  if (st != DEC_OK) return st;
  if ((reinterpret_cast<uintptr_t>(error_word) & 3u) != 0)
    return decattn::record_error(DEC_ERR_INVALID_ARG, "error_word must be 4-byte aligned");
  if ((st = decattn::check_reachable(error_word, "error_word")) != DEC_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 7 * sizeof(uint32_t), s) != cudaSuccess) {
    (void)cudaGetLastError();
    return decattn::record_error(DEC_ERR_CUDA, "clearing the scratch header failed");
  }
  st = dec_gqa_decode_attn(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale,
                           num_parts, scratch, kNoAllocScratchBytes, stream);
  if (st != DEC_OK || error_word == nullptr) return st;
  // the error word sits at byte 0 of the scratch; hand this call's value to the caller
  if (cudaMemcpyAsync(error_word, scratch, sizeof(uint32_t), cudaMemcpyDefault, s) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return decattn::record_error(DEC_ERR_CUDA, "copying the error word out failed");
  }
  return DEC_OK;
}
