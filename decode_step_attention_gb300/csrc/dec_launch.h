// Internal launchers of the decode-step attention kernels (host side). Arguments
// are already validated by the C-ABI layer in api.cu; each launcher only enqueues
// its kernel and returns cudaGetLastError().
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "decattn.h"

namespace decattn {

// Store a one-line reason for dec_last_error() on this thread and return `status`.
dec_status record_error(dec_status status, const char *message);

constexpr size_t kWorkspaceHeaderBytes = 256;
constexpr int kSplitTile = 64;     // tokens per pipeline stage of the split pass
constexpr int kSplitMaxB = 8192;   // largest batch the split pass keeps prefix sums for
constexpr int kSplitMaxG = 8;      // largest query-head group per KV head

cudaError_t launch_rmsnorm_residual(const void *x, void *residual, const void *weight, void *y,
                                    int B, int hidden, float eps, cudaStream_t stream);

cudaError_t launch_qknorm_rope_append(void *q, const void *k_new, const void *v_new,
                                      const void *q_norm_w, const void *k_norm_w, void *k_cache,
                                      void *v_cache, const int32_t *pos, int B, int Hq, int Hkv,
                                      int D, int T_cap, double theta, int interleaved, float eps,
                                      uint32_t *error_word, cudaStream_t stream);

// Split pass geometry: bytes of dynamic shared memory and CTAs resident per SM.
size_t split_smem_bytes(int D, int B);
int split_ctas_per_sm(int D, int B, int device);

cudaError_t launch_gqa_split(const CUtensorMap &kmap, const CUtensorMap &vmap, const void *q,
                             const int32_t *lens, int B, int Hq, int Hkv, int D, int T_cap,
                             float scale_log2, int num_parts, void *workspace,
                             cudaStream_t stream);

cudaError_t launch_split_merge(const void *workspace, const int32_t *lens, void *out, int B,
                               int Hq, int Hkv, int D, int T_cap, int num_parts,
                               cudaStream_t stream);

}  // namespace decattn
