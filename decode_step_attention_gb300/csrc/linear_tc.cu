// Projections on either side of the block: Y[B, N] = X[B, K] W[N, K]^T (+ R[B, N]),
// bf16 in and out, fp32 accumulation, on the 5th-generation tensor cores (tcgen05,
// accumulator in tensor memory). The packed QKV projection feeds the rotation step and
// the output projection adds the residual stream in its epilogue (cutileGPT README,
// "The current runtime includes": packed QKV projections, fused down-projection +
// residual epilogues). The weight is stored one row per output feature, the B[N, K]
// layout of the PyGPUkit 0.2.18 page ("Optimized BF16 GEMV").
//
// Decode batches are small, so the roles are swapped: the MMA's M dimension runs over
// 128 output features (rows of W) and its N dimension over a tile of NB batch rows,
//   D[n, b] = sum_k W[n, k] X[b, k]      (tcgen05.mma kind::f16, M = 128, N = NB)
// with both operands K-major in 128-byte-swizzled shared memory, loaded by TMA into a
// ring of stages. A CTA owns one 128 x NB output tile and a contiguous slice of the
// K chunks; when the output tiles alone would leave SMs idle, K is split over several
// CTAs and a second kernel sums their fp32 partials in slice order, so the result does
// not depend on timing.
//
// Warps: 0-3 epilogue (warp w reads tensor-memory lanes 32w .. 32w + 31), 4 TMA
// producer, 5 MMA issuer. Every wait is bounded in time; a stalled pipeline sets an
// error bit and the CTA still releases its tensor memory.
#include <algorithm>

#include "dec_device.cuh"
#include "dec_launch.h"

namespace decattn {
namespace {

constexpr int kLinM = 128;      // output features per tile (MMA M)
constexpr int kLinKChunk = 64;  // K elements per stage: one 128-byte swizzle row
constexpr int kLinThreads = 192;
constexpr int kLinMaxSplits = 64;

template <int NB>
struct LinGeom {
  static constexpr int kWBytes = kLinM * kLinKChunk * 2;  // 16 KB
  static constexpr int kXBytes = NB * kLinKChunk * 2;     // a multiple of 1 KB for NB >= 8
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kStages = NB >= 256 ? 4 : 6;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes;  // + alignment pad
  static constexpr uint32_t kTmemCols = NB < 32 ? 32 : NB;  // a power of two >= 32
};

// ---- tcgen05 helpers (inline PTX) ----------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand stored as 128-byte swizzle atoms
// (8 rows x 128 bytes): start address, the stride between 8-row groups (1024 bytes),
// the descriptor version bit and the swizzle mode (2 = 128-byte). The leading-offset
// field is not used by this layout.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5), bf16 A (7-9) and
// B (10-12), both K-major (bits 15, 16 clear), N >> 3 (17-22), M >> 4 (24-28).
constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// This thread's tensor-memory lane, 16 consecutive fp32 columns from `taddr`.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void set_error(uint32_t *error_word, uint32_t bit) {
  if (error_word != nullptr) atomicOr(error_word, bit);
}

// grid (N / 128, ceil(B / NB), S). Tile: features [128 x, +128), batch rows [NB y, +NB),
// K chunks [z cps, min((z + 1) cps, nchunks)). With `partial` set, the fp32 tile goes to
// slice z of the partial buffer [S, B, N]; otherwise y = bf16(tile (+ residual)).
template <int NB>
__global__ void __launch_bounds__(kLinThreads, 1) linear_tc_kernel(
    const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
    const __nv_bfloat16 *residual, __nv_bfloat16 *y, float *__restrict__ partial, int B, int N,
    int nchunks, int cps, uint32_t *error_word) {
  using G = LinGeom<NB>;
  constexpr int S = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_bar[2 * S + 1];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar_full = smem_addr(&s_bar[0]);
  const uint32_t bar_empty = bar_full + 8 * S;
  const uint32_t bar_acc = bar_empty + 8 * S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kLinM, b0 = blockIdx.y * NB;
  const int c_begin = blockIdx.z * cps;
  const int c_end = min(c_begin + cps, nchunks);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(&s_tmem), G::kTmemCols);
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();
  pdl_wait_prior_grid();

  if (warp == 4) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t w_policy = l2_policy_evict_first();  // each weight byte is read once
      const uint64_t x_policy = l2_policy_evict_last();   // X is read by every feature tile
      int issued = 0;
      for (int c = c_begin; c < c_end; ++c, ++issued) {
        const int st = issued % S, round = issued / S;
        if (s_abort) break;
        if (round > 0 && !mbar_wait_bounded(bar_empty + 8 * st, (round - 1) & 1)) {
          set_error(error_word, kErrWaitTimeout);
          s_abort = 1;
          break;
        }
        const uint32_t full = bar_full + 8 * st;
        const uint32_t ws = s_base + st * G::kStageBytes;
        mbar_arrive_expect_tx(full, G::kStageBytes);
        tma_load_2d(ws, &wmap, c * kLinKChunk, n0, full, w_policy);
        tma_load_2d(ws + G::kWBytes, &xmap, c * kLinKChunk, b0, full, x_policy);
      }
      // Do not leave while a copy into this CTA's shared memory is still in flight.
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
        if (!mbar_wait_bounded(bar_full + 8 * (j % S), (j / S) & 1)) {
          set_error(error_word, kErrWaitTimeout);
          break;
        }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kLinM, NB);
      int done = 0;
      for (int c = c_begin; c < c_end; ++c, ++done) {
        const int st = done % S, round = done / S;
        if (s_abort || !mbar_wait_bounded(bar_full + 8 * st, round & 1)) {
          set_error(error_word, kErrWaitTimeout);
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t ws = s_base + st * G::kStageBytes;
#pragma unroll
        for (int k = 0; k < kLinKChunk / 16; ++k)
          umma_bf16(tmem, smem_desc_sw128(ws + 32 * k), smem_desc_sw128(ws + G::kWBytes + 32 * k),
                    idesc, (done > 0 || k > 0) ? 1u : 0u);
        umma_commit(bar_empty + 8 * st);  // the stage is free once these MMAs have read it
      }
      umma_commit(bar_acc);  // the accumulator is final once everything above completes
      mbar_wait_bounded(bar_acc, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue, warps 0-3
    const bool acc_done = __all_sync(0xffffffffu, mbar_wait_bounded(bar_acc, 0) ? 1 : 0);
    const bool ready = acc_done && !s_abort && c_end > c_begin;
    tc_fence_after();
    if (ready) {
      const int n = n0 + 32 * warp + lane;  // this thread's output feature
      const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
      for (int cb = 0; cb < NB; cb += 16) {
        if (b0 + cb >= B) break;
        float v[16];
        tmem_ld16(trow + cb, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int b = b0 + cb + j;
          if (b < B) {
            if (partial != nullptr) {
              partial[((size_t)blockIdx.z * B + b) * N + n] = v[j];
            } else {
              float r = v[j];
              if (residual != nullptr) r += __bfloat162float(residual[(size_t)b * N + n]);
              y[(size_t)b * N + n] = __float2bfloat16_rn(r);
            }
          }
        }
      }
    } else if (lane == 0 && !acc_done) {
      set_error(error_word, kErrWaitTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }
}

// y = bf16(sum over slices s = 0 .. S-1 of partial[s] (+ residual)), in slice order.
__global__ void __launch_bounds__(256) linear_reduce_kernel(const float4 *__restrict__ partial,
                                                            const __nv_bfloat16 *residual,
                                                            __nv_bfloat16 *y, size_t total4,
                                                            int S) {
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 acc = partial[i];
    for (int s = 1; s < S; ++s) {
      const float4 p = partial[(size_t)s * total4 + i];
      acc.x += p.x;
      acc.y += p.y;
      acc.z += p.z;
      acc.w += p.w;
    }
    if (residual != nullptr) {
      const uint2 rr = reinterpret_cast<const uint2 *>(residual)[i];
      acc.x += bf16_lo(rr.x);
      acc.y += bf16_hi(rr.x);
      acc.z += bf16_lo(rr.y);
      acc.w += bf16_hi(rr.y);
    }
    reinterpret_cast<uint2 *>(y)[i] =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

template <int NB>
cudaError_t launch_linear_nb(const CUtensorMap &wmap, const CUtensorMap &xmap,
                             const void *residual, void *y, float *partial, int B, int N, int K,
                             int splits, uint32_t *error_word, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = LinGeom<NB>::kSmem;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(linear_tc_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  const int nchunks = K / kLinKChunk;
  const int cps = (nchunks + splits - 1) / splits;
  const dim3 grid(N / kLinM, (B + NB - 1) / NB, splits);
  auto *rp = static_cast<const __nv_bfloat16 *>(residual);
  auto *yp = static_cast<__nv_bfloat16 *>(y);
  e = launch_pdl(linear_tc_kernel<NB>, grid, dim3(kLinThreads), smem, stream, wmap, xmap, rp, yp,
                 splits > 1 ? partial : nullptr, B, N, nchunks, cps, error_word);
  if (e != cudaSuccess) return e;
  if (splits > 1) {
    const size_t total4 = (size_t)B * N / 4;
    const int blocks = (int)std::min<size_t>((total4 + 255) / 256, 4 * 152);
    e = launch_pdl(linear_reduce_kernel, dim3(blocks), dim3(256), 0, stream,
                   reinterpret_cast<const float4 *>(partial), rp, yp, total4, splits);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

int linear_batch_tile(int B) {
  return B <= 16 ? 16 : B <= 32 ? 32 : B <= 64 ? 64 : B <= 128 ? 128 : 256;
}

// K splits for a (B, N, K) projection on `sm_count` SMs, at most `max_splits`: the count
// that minimises (waves of CTAs) x (chunks per CTA) plus a fixed cost for the reduce
// launch and the partials' round trip, counted in chunk-loads. Every slice is non-empty.
int linear_splits(int B, int N, int K, int sm_count, int max_splits) {
  const int nb = linear_batch_tile(B);
  const long long tiles = (long long)(N / kLinM) * ((B + nb - 1) / nb);
  const int nchunks = K / kLinKChunk;
  const double chunk_bytes = (double)sm_count * (kLinM * kLinKChunk * 2);
  auto waves = [&](long long ctas) { return (ctas + sm_count - 1) / sm_count; };
  int best = 1;
  double best_cost = (double)waves(tiles) * nchunks;
  const int cap = std::min(std::min(max_splits, kLinMaxSplits), nchunks);
  for (int s = 2; s <= cap; ++s) {
    const int cps = (nchunks + s - 1) / s;
    if ((nchunks + cps - 1) / cps != s) continue;  // that split would leave a slice empty
    const double cost = (double)waves(tiles * s) * cps + 4.0 +
                        2.0 * s * (double)B * N * 4.0 / chunk_bytes;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

cudaError_t launch_linear(const CUtensorMap &wmap, const CUtensorMap &xmap, const void *residual,
                          void *y, float *partial, int B, int N, int K, int splits,
                          uint32_t *error_word, cudaStream_t stream) {
  switch (linear_batch_tile(B)) {
    case 16:
      return launch_linear_nb<16>(wmap, xmap, residual, y, partial, B, N, K, splits, error_word,
                                  stream);
    case 32:
      return launch_linear_nb<32>(wmap, xmap, residual, y, partial, B, N, K, splits, error_word,
                                  stream);
    case 64:
      return launch_linear_nb<64>(wmap, xmap, residual, y, partial, B, N, K, splits, error_word,
                                  stream);
    case 128:
      return launch_linear_nb<128>(wmap, xmap, residual, y, partial, B, N, K, splits, error_word,
                                   stream);
    default:
      return launch_linear_nb<256>(wmap, xmap, residual, y, partial, B, N, K, splits, error_word,
                                   stream);
  }
}

}  // namespace decattn
