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
// ring of stages; each stage holds several 64-wide K pieces of the same weight rows, so
// a row's consecutive bytes are requested together.
//
// Split K without a round trip through HBM: the S CTAs that share one output tile (one
// K slice each) form a thread-block cluster. Each CTA moves its accumulator from tensor
// memory to its own shared memory; after a cluster barrier, CTA r sums part r/S of the
// tile over all S CTAs' shared memory (distributed shared memory reads, in CTA order,
// so the result does not depend on timing), adds the residual and stores bf16.
//
// Warps: 0-3 move the accumulator out (warp w reads tensor-memory lanes 32w .. 32w+31),
// 4 is the TMA producer, 5 issues the MMAs; all six reduce and store. Every mbarrier
// wait is bounded in time; a stalled pipeline sets an error bit, and every CTA still
// reaches both cluster barriers and releases its tensor memory.
#include <algorithm>
#include <atomic>

#include "dec_device.cuh"
#include "dec_launch.h"
#include "rope_angles.cuh"

namespace decattn {
namespace {

constexpr int kLinM = 128;      // output features per tile (MMA M)
constexpr int kLinSub = 64;     // K elements per piece: one 128-byte swizzle row
constexpr int kLinThreads = 192;

// Stage layout: kSub pieces of W (16 KB each), then kSub pieces of X; with the RMSNorm
// prologue (kNorm), then kSub pieces of the residual R and kSub 128-byte pieces of the
// norm weight, the stage rounded up to 1 KB (the swizzled pieces need 1 KB alignment).
template <int NB, bool kNorm = false>
struct LinGeom {
  static constexpr int kSub = (kNorm ? NB >= 128 : NB >= 256) ? 1 : 2;  // K pieces per stage
  static constexpr int kWSub = kLinM * kLinSub * 2;        // 16 KB
  static constexpr int kXSub = NB * kLinSub * 2;           // a multiple of 1 KB
  static constexpr int kRSub = kNorm ? kXSub : 0;          // the residual's piece
  static constexpr int kNSub = kNorm ? kLinSub * 2 : 0;    // the norm weight's piece
  static constexpr int kSubBytes = kWSub + kXSub + kRSub + kNSub;
  static constexpr int kROff = kSub * (kWSub + kXSub);     // R pieces within a stage
  static constexpr int kNOff = kROff + kSub * kRSub;       // norm-weight pieces
  static constexpr int kStageBytes = (kSub * kSubBytes + 1023) / 1024 * 1024;
  static constexpr int kNormStages = (196 * 1024) / kStageBytes;
  static constexpr int kStages =
      kNorm ? (kNormStages > 8 ? 8 : kNormStages)
            : (NB == 16 ? 6 : NB == 32 ? 5 : NB == 128 ? 3 : 4);
  static constexpr size_t kRing = (size_t)kStages * kStageBytes;
  static constexpr size_t kAcc = (size_t)kLinM * NB * 4;   // fp32 tile, [NB][128]
  static constexpr size_t kSmem = 1024 + (kRing > kAcc ? kRing : kAcc);
  static constexpr uint32_t kTmemCols = NB < 32 ? 32 : NB;  // a power of two >= 32
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kStages >= 2, "pipeline depth");
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

// ---- cluster helpers ------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The barrier before a CTA exits, so that no CTA leaves while another still reads its
// shared memory. Execution order is all it needs: every remote load of the arriving thread
// has returned (its value has been used), so the arrival is relaxed. A release here would
// also wait for the thread's global stores to be acknowledged.
__device__ __forceinline__ void cluster_exit_sync() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
               "barrier.cluster.wait.aligned;" ::: "memory");
}

// The address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// The sum over the cluster's first S CTAs (S <= 8), in CTA order, of the float4 at
// shared address `addr`: every load is issued before the first add, so the remote
// latencies overlap instead of adding up.
__device__ __forceinline__ float4 cluster_sum_f4(uint32_t addr, uint32_t S) {
  float4 p[8];
#pragma unroll
  for (uint32_t q = 0; q < 8; ++q)
    if (q < S) p[q] = ld_cluster_f4(cluster_map(addr, q));
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (uint32_t q = 0; q < 8; ++q)
    if (q < S) {
      a.x += p[q].x;
      a.y += p[q].y;
      a.z += p[q].z;
      a.w += p[q].w;
    }
  return a;
}

__device__ __forceinline__ uint4 ld_smem_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_smem_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void set_error(uint32_t *error_word, uint32_t bit) {
  if (error_word != nullptr) atomicOr(error_word, bit);
}

// The rotation epilogue of the packed QKV projection (head_dim 128). Feature tile
// blockIdx.x is one head: q heads first, then k heads, then v heads. Batch column c of
// the tile goes to CTA c mod S of the cluster and, there, to one warp; lane j holds
// features 4j .. 4j+3, the sum of the S slices' accumulators. q and k heads: optional
// RMSNorm over the head (a warp reduction), then RoPE at pos[b] (NeoX partners 16
// lanes apart, interleaved partners in the lane); q goes to q_out, k to cache slot
// pos[b]; v heads are copied to their slot. The arithmetic follows the standalone
// rotation kernel, on the unrounded projection instead of its bf16 copy.
template <int NB>
__device__ void qkv_rot_epilogue(const QkvRotArgs &rot, const unsigned long long *turns,
                                 uint32_t acc_addr, uint32_t S, uint32_t rank, int b0, int B,
                                 const float *col_scale, uint32_t *error_word) {
  constexpr int kD = 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x;
  const int kind = head < rot.Hq ? 0 : head < rot.Hq + rot.Hkv ? 1 : 2;
  const int hh = kind == 0 ? head : kind == 1 ? head - rot.Hq : head - rot.Hq - rot.Hkv;
  const int step = (int)S * (kLinThreads / 32);
  for (int c = (int)rank + (int)S * warp; c < NB; c += step) {
    const int b = b0 + c;
    if (b >= B) break;
    const int i4 = c * (kLinM / 4) + lane;
    const float4 a = cluster_sum_f4(acc_addr + 16u * i4, S);
    const float cs0 = col_scale != nullptr ? col_scale[c] : 1.f;
    float x[4] = {a.x * cs0, a.y * cs0, a.z * cs0, a.w * cs0};
    const int p = rot.pos[b];
    if (p < 0 || p >= rot.T_cap) {
      if (lane == 0 && head == 0) set_error(error_word, kErrPosSkipped);
      continue;
    }
    const int e0 = 4 * lane;
    if (kind < 2) {
      const auto *nw = static_cast<const __nv_bfloat16 *>(kind == 0 ? rot.q_norm_w : rot.k_norm_w);
      if (nw != nullptr) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(x[e], x[e], ss);
        ss = warp_sum(ss);
        const float rstd = rsqrtf(ss * (1.0f / (float)kD) + rot.eps);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = x[e] * rstd * __bfloat162float(nw[e0 + e]);
      }
      // the column's 64 angles: lane l forms those of pairs l and l + 32, the others
      // read them with shuffles
      float s_lo, c_lo, s_hi, c_hi;
      rope_sincos_turns(p, turns[lane], s_lo, c_lo);
      rope_sincos_turns(p, turns[lane + 32], s_hi, c_hi);
      auto angle = [&](int i, float &sn, float &cs) {
        const float sl = __shfl_sync(0xffffffffu, s_lo, i & 31);
        const float sh = __shfl_sync(0xffffffffu, s_hi, i & 31);
        const float cl = __shfl_sync(0xffffffffu, c_lo, i & 31);
        const float ch = __shfl_sync(0xffffffffu, c_hi, i & 31);
        sn = i < 32 ? sl : sh;
        cs = i < 32 ? cl : ch;
      };
      float yv[4];
      if (!rot.interleaved) {
        // NeoX: feature d < 64 pairs with d + 64, which lives 16 lanes away
        const bool first = lane < 16;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
          float sn, cs;
          angle((lane & 15) * 4 + e, sn, cs);
          yv[e] = first ? (x[e] * cs - other * sn) : (other * sn + x[e] * cs);
        }
      } else {
        // interleaved: feature 2i pairs with 2i + 1, both in this lane
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          float sn, cs;
          angle((e0 + e) >> 1, sn, cs);
          yv[e] = x[e] * cs - x[e + 1] * sn;
          yv[e + 1] = x[e] * sn + x[e + 1] * cs;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = yv[e];
    }
    const uint2 packed = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    __nv_bfloat16 *dst;
    if (kind == 0) {
      dst = static_cast<__nv_bfloat16 *>(rot.q_out) + ((size_t)b * rot.Hq + hh) * kD;
    } else {
      const size_t slot = (((size_t)b * rot.Hkv + hh) * rot.T_cap + p) * kD;
      dst = static_cast<__nv_bfloat16 *>(kind == 1 ? rot.k_cache : rot.v_cache) + slot;
    }
    *reinterpret_cast<uint2 *>(dst + e0) = packed;
  }
}

// The RMSNorm prologue applied to one activation piece in place (warps 0-3): the piece
// holds NB rows of 64 values of x, the residual's piece the same rows of r, both in the
// 128-byte swizzle (16-byte chunk c of row j sits at chunk c ^ (j & 7)); wsm holds the
// piece's 64 norm weights.
// Thread t takes physical chunk t & 7 of rows t / 8 + 16 m: u = bf16((x + r) * w) goes
// back over x for the MMA, the squares of the fp32 sums go to ss[m], and the CTAs of
// the first feature tile store h = bf16(x + r).
template <int NB>
__device__ __forceinline__ void norm_piece(uint32_t xs, uint32_t rs, uint32_t wsm,
                                           const LinNorm &norm, int k_base, int b0, int B, int K,
                                           bool write_h, float (&ss)[NB / 16]) {
  const int t = threadIdx.x;  // 0 .. 127
  const int pc = t & 7;
  __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(norm.h_out);
#pragma unroll
  for (int m = 0; m < NB / 16; ++m) {
    const int row = (t >> 3) + 16 * m;
    const int lc = pc ^ (row & 7);  // logical chunk: K offset lc * 8 in the piece
    const int k0 = k_base + lc * 8;
    const uint32_t off = (uint32_t)(row * 128 + pc * 16);
    const uint4 xv = ld_smem_u4(xs + off);
    const uint4 rv = norm.has_r ? ld_smem_u4(rs + off) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 wv = ld_smem_u4(wsm + lc * 16);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t uo[4], ho[4];
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float s0 = bf16_lo(xw[e]) + bf16_lo(rw[e]);
      const float s1 = bf16_hi(xw[e]) + bf16_hi(rw[e]);
      acc = fmaf(s0, s0, acc);
      acc = fmaf(s1, s1, acc);
      uo[e] = pack_bf16x2(s0 * bf16_lo(ww[e]), s1 * bf16_hi(ww[e]));
      ho[e] = pack_bf16x2(s0, s1);
    }
    ss[m] += acc;
    st_smem_u4(xs + off, make_uint4(uo[0], uo[1], uo[2], uo[3]));
    if (write_h && b0 + row < B)
      *reinterpret_cast<uint4 *>(h + (size_t)(b0 + row) * K + k0) =
          make_uint4(ho[0], ho[1], ho[2], ho[3]);
  }
}

// grid (N / 128, ceil(B / NB), S), cluster (1, 1, S). Tile: features [128 x, +128),
// batch rows [NB y, +NB); K pieces [z cps, min((z + 1) cps, nsub)) of 64 each.
// kRot: the packed QKV projection with head_dim 128, whose epilogue is the rotation
// step (QK-norm, RoPE, K/V append) instead of a plain store. kNorm: the operand is
// RMSNorm(x + r) formed in the pipeline (LinNorm), warps 0-3 transforming each stage
// between its copy and its MMAs.
template <int NB, bool kRot, bool kNorm>
__global__ void __launch_bounds__(kLinThreads, 1) linear_tc_kernel(
    const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
    const __grid_constant__ CUtensorMap rmap, const __nv_bfloat16 *residual,
    __nv_bfloat16 *y, int B, int N, int nsub, int cps,
    uint32_t *error_word, const LinNorm norm, const __grid_constant__ QkvRotArgs rot) {
  using G = LinGeom<NB, kNorm>;
  constexpr int S = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_bar[3 * S + 1];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ unsigned long long s_turns[kRot ? 64 : 1];
  __shared__ float s_ss[kNorm ? NB : 1];     // this CTA's sums of squares per batch row
  __shared__ float s_scale[kNorm ? NB : 1];  // rsqrt(mean square + eps) per batch row

  // 1024-byte aligned in the shared window; indexing off the __shared__ array keeps the
  // compiler's knowledge that this is shared memory (shared loads and stores rather than
  // generic ones)
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float *acc_s = reinterpret_cast<float *>(smem);  // [NB][128] after the main loop
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar_full = smem_addr(&s_bar[0]);
  const uint32_t bar_empty = bar_full + 8 * S;
  const uint32_t bar_ready = bar_empty + 8 * S;  // kNorm: the stage's operand is formed
  const uint32_t bar_acc = bar_ready + 8 * S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kLinM, b0 = blockIdx.y * NB;
  const int c_begin = blockIdx.z * cps;
  const int c_end = min(c_begin + cps, nsub);
  const int nstage = (c_end - c_begin + G::kSub - 1) / G::kSub;

  if constexpr (kRot) {
    if (threadIdx.x < 64) s_turns[threadIdx.x] = rot.turns[threadIdx.x];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_ready + 8 * s, 128);
    }
    mbar_init(bar_acc, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(&s_tmem), G::kTmemCols);
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
    if (kNorm && norm.has_r) tma_prefetch_desc(&rmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();
  const uint64_t w_policy = l2_policy_evict_first();  // each weight byte is read once
  const bool with_r = kNorm && norm.has_r;
  auto stage_tx = [&](int nv) {
    return (uint32_t)(nv * (G::kWSub + G::kXSub + G::kNSub + (with_r ? G::kRSub : 0)));
  };
  // No kernel that may run ahead of this one's wait writes a weight (only this library's
  // kernels let a successor start early), so the first ring's weight pieces are requested
  // before the wait: their HBM latency overlaps the previous kernel's tail. Each stage's
  // barrier expects the whole stage; the activation pieces follow after the wait.
  const int pre = min(nstage, S);
  if (warp == 4 && lane == 0) {
    for (int i = 0; i < pre; ++i) {
      const int c0 = c_begin + i * G::kSub;
      const int nv = min(G::kSub, c_end - c0);
      const uint32_t full = bar_full + 8 * i;
      mbar_arrive_expect_tx(full, stage_tx(nv));
      for (int j = 0; j < nv; ++j)
        tma_load_2d(s_base + i * G::kStageBytes + j * G::kWSub, &wmap, (c0 + j) * kLinSub, n0,
                    full, w_policy);
    }
  }
  pdl_wait_prior_grid();

  if (warp == 4) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t x_policy = l2_policy_evict_last();   // X is read by every feature tile
      int issued = 0;
      for (; issued < nstage; ++issued) {
        const int st = issued % S, round = issued / S;
        const int c0 = c_begin + issued * G::kSub;
        const int nv = min(G::kSub, c_end - c0);
        const uint32_t full = bar_full + 8 * st;
        const uint32_t ws = s_base + st * G::kStageBytes;
        if (round > 0) {  // the first round's weights are already on their way
          if (s_abort) break;
          if (!mbar_wait_bounded(bar_empty + 8 * st, (round - 1) & 1)) {
            set_error(error_word, kErrWaitTimeout);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(full, stage_tx(nv));
          for (int j = 0; j < nv; ++j)
            tma_load_2d(ws + j * G::kWSub, &wmap, (c0 + j) * kLinSub, n0, full, w_policy);
        }
        for (int j = 0; j < nv; ++j) {
          tma_load_2d(ws + G::kSub * G::kWSub + j * G::kXSub, &xmap, (c0 + j) * kLinSub, b0, full,
                      x_policy);
          if constexpr (kNorm) {
            if (with_r)
              tma_load_2d(ws + G::kROff + j * G::kRSub, &rmap, (c0 + j) * kLinSub, b0, full,
                          x_policy);
            bulk_load(ws + G::kNOff + j * G::kNSub,
                      static_cast<const __nv_bfloat16 *>(norm.norm_w) + (c0 + j) * kLinSub,
                      G::kNSub, full);
          }
        }
      }
      // Do not move on while a copy into this CTA's shared memory is still in flight.
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
      for (int i = 0; i < nstage; ++i) {
        const int st = i % S, round = i / S;
        // with the prologue the stage is ready once warps 0-3 have formed its operand
        const uint32_t gate = (kNorm ? bar_ready : bar_full) + 8 * st;
        if (s_abort || !mbar_wait_bounded(gate, round & 1)) {
          set_error(error_word, kErrWaitTimeout);
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const int nv = min(G::kSub, c_end - (c_begin + i * G::kSub));
        const uint32_t ws = s_base + st * G::kStageBytes;
        for (int j = 0; j < nv; ++j) {
          const uint32_t wa = ws + j * G::kWSub, xa = ws + G::kSub * G::kWSub + j * G::kXSub;
#pragma unroll
          for (int k = 0; k < kLinSub / 16; ++k)
            umma_bf16(tmem, smem_desc_sw128(wa + 32 * k), smem_desc_sw128(xa + 32 * k), idesc,
                      (i > 0 || j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(bar_empty + 8 * st);  // the stage is free once these MMAs have read it
      }
      umma_commit(bar_acc);  // the accumulator is final once everything above completes
      mbar_wait_bounded(bar_acc, 0);
    }
  } else {
    if constexpr (kNorm) {
      // ------------------------------------- the RMSNorm prologue, stage by stage
      float ss[NB / 16];
#pragma unroll
      for (int m = 0; m < NB / 16; ++m) ss[m] = 0.f;
      const int K = nsub * kLinSub;
      const bool write_h = norm.h_out != nullptr && blockIdx.x == 0;
      for (int i = 0; i < nstage; ++i) {
        const int st = i % S, round = i / S;
        if (s_abort || !mbar_wait_bounded(bar_full + 8 * st, round & 1)) {
          set_error(error_word, kErrWaitTimeout);
          s_abort = 1;
          break;
        }
        const uint32_t ws = s_base + st * G::kStageBytes;
        const int c0 = c_begin + i * G::kSub;
        const int nv = min(G::kSub, c_end - c0);
        for (int j = 0; j < nv; ++j)
          norm_piece<NB>(ws + G::kSub * G::kWSub + j * G::kXSub, ws + G::kROff + j * G::kRSub,
                         ws + G::kNOff + j * G::kNSub, norm, (c0 + j) * kLinSub, b0, B, K,
                         write_h, ss);
        fence_proxy_async_smem();  // the MMAs read the operand through the async proxy
        mbar_arrive(bar_ready + 8 * st);
      }
      // per row: the 8 threads of a row hold its partial sums
#pragma unroll
      for (int m = 0; m < NB / 16; ++m) {
        float v = ss[m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if ((threadIdx.x & 7) == 0) s_ss[(threadIdx.x >> 3) + 16 * m] = v;
      }
    }
    // ------------------------------------------- accumulator -> shared memory (warps 0-3)
    const bool acc_done = __all_sync(0xffffffffu, mbar_wait_bounded(bar_acc, 0) ? 1 : 0);
    tc_fence_after();
    if (acc_done && !s_abort) {
      const int row = 32 * warp + lane;  // feature n0 + row
      const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
      for (int cb = 0; cb < NB; cb += 16) {
        float v[16];
        tmem_ld16(trow + cb, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc_s[(cb + j) * kLinM + row] = v[j];  // conflict-free
      }
    } else if (lane == 0) {
      set_error(error_word, kErrWaitTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }
  // ---------------------------------------------------------- cluster-wide reduction
  cluster_sync();  // every slice's accumulator is in its CTA's shared memory
  const uint32_t S_ = gridDim.z;
  const uint32_t rank = blockIdx.z;
  const float *col_scale = nullptr;
  if constexpr (kNorm) {
    // each batch row's sum of squares over the whole K: the slices' sums, in CTA order
    const uint32_t ss_addr = smem_addr(s_ss);
    for (int c = threadIdx.x; c < NB; c += kLinThreads) {
      float p[8];
#pragma unroll
      for (uint32_t q = 0; q < 8; ++q)
        if (q < S_) p[q] = ld_cluster_f32(cluster_map(ss_addr + 4u * c, q));
      float tot = 0.f;
#pragma unroll
      for (uint32_t q = 0; q < 8; ++q)
        if (q < S_) tot += p[q];
      s_scale[c] = rsqrtf(tot * norm.inv_k + norm.eps);
    }
    __syncthreads();
    col_scale = s_scale;
  }
  if constexpr (kRot) {
    qkv_rot_epilogue<NB>(rot, s_turns, smem_addr(acc_s), S_, rank, b0, B, col_scale,
                         error_word);
    cluster_exit_sync();  // no CTA leaves while another still reads its shared memory
    return;
  }
  constexpr int Q = kLinM * NB / 4;  // float4s in the tile
  const int q0 = (int)((uint64_t)Q * rank / S_), q1 = (int)((uint64_t)Q * (rank + 1) / S_);
  const uint32_t acc_addr = smem_addr(acc_s);
  // four float4s per thread per round, so their remote loads are in flight together
  constexpr int kU = 4;
  for (int i0 = q0 + threadIdx.x; i0 < q1; i0 += kU * kLinThreads) {
    float4 a[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * kLinThreads;
      if (i < q1 && b0 + i / (kLinM / 4) < B) a[u] = cluster_sum_f4(acc_addr + 16u * i, S_);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * kLinThreads;
      const int c = i / (kLinM / 4);          // batch column of the tile
      const int row = (i % (kLinM / 4)) * 4;  // first of four features
      const int b = b0 + c;
      if (i >= q1 || b >= B) continue;
      float4 v = a[u];
      if (col_scale != nullptr) {
        const float cs = col_scale[c];
        v.x *= cs;
        v.y *= cs;
        v.z *= cs;
        v.w *= cs;
      }
      const size_t o = (size_t)b * N + n0 + row;
      if (residual != nullptr) {
        const uint2 rr = *reinterpret_cast<const uint2 *>(residual + o);
        v.x += bf16_lo(rr.x);
        v.y += bf16_hi(rr.x);
        v.z += bf16_lo(rr.y);
        v.w += bf16_hi(rr.y);
      }
      *reinterpret_cast<uint2 *>(y + o) =
          make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
  }
  cluster_exit_sync();  // no CTA leaves while another still reads its shared memory
}

// ---- host side ---------------------------------------------------------------------
constexpr int kMaxDev = 64;
constexpr int kMaxCluster = 8;

template <int NB, bool kRot, bool kNorm>
cudaError_t ensure_attr(int dev) {
  static std::atomic<bool> done[kMaxDev];
  if (dev >= 0 && dev < kMaxDev && done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<NB, kRot, kNorm>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)LinGeom<NB, kNorm>::kSmem);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev].store(true);
  return e;
}

cudaLaunchConfig_t cluster_config(dim3 grid, size_t smem, cudaStream_t stream, int splits,
                                  cudaLaunchAttribute (&attr)[2], bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kLinThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)splits;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

// Clusters of `splits` CTAs that fit on the device at once (cached per device).
template <int NB, bool kNorm>
int resident_clusters(int dev, int splits) {
  static std::atomic<int> cache[kMaxDev][kMaxCluster + 1];
  if (dev >= 0 && dev < kMaxDev) {
    const int c = cache[dev][splits].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (ensure_attr<NB, false, kNorm>(dev) == cudaSuccess) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(dim3(1, 1, splits), LinGeom<NB, kNorm>::kSmem,
                                            nullptr, splits, attr, false);
    if (cudaOccupancyMaxActiveClusters(&n, linear_tc_kernel<NB, false, kNorm>, &cfg) !=
        cudaSuccess)
      n = 0;
  }
  if (n <= 0) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (n > 0 && dev >= 0 && dev < kMaxDev) cache[dev][splits].store(n);
  return n;
}

template <bool kNorm>
int resident(int nb, int dev, int splits) {
  switch (nb) {
    case 16: return resident_clusters<16, kNorm>(dev, splits);
    case 32: return resident_clusters<32, kNorm>(dev, splits);
    case 64: return resident_clusters<64, kNorm>(dev, splits);
    case 128: return resident_clusters<128, kNorm>(dev, splits);
    default: return resident_clusters<256, kNorm>(dev, splits);
  }
}

// Everything a launch passes besides the tensor maps and the shape.
struct LinLaunch {
  const CUtensorMap *rmap;  // the residual's map (kNorm; any valid map otherwise)
  const void *residual;
  void *y;
  LinNorm norm;
  QkvRotArgs rot;
};

template <int NB, bool kRot, bool kNorm>
cudaError_t launch_linear_nb(const CUtensorMap &wmap, const CUtensorMap &xmap,
                             const LinLaunch &L, int B, int N, int K, int splits,
                             uint32_t *error_word, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = ensure_attr<NB, kRot, kNorm>(dev)) != cudaSuccess) return e;
  const int nsub = K / kLinSub;
  const int cps = (nsub + splits - 1) / splits;
  const dim3 grid(N / kLinM, (B + NB - 1) / NB, splits);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg =
      cluster_config(grid, LinGeom<NB, kNorm>::kSmem, stream, splits, attr, true);
  e = cudaLaunchKernelEx(&cfg, linear_tc_kernel<NB, kRot, kNorm>, wmap, xmap, *L.rmap,
                         static_cast<const __nv_bfloat16 *>(L.residual),
                         static_cast<__nv_bfloat16 *>(L.y), B, N, nsub, cps,
                         error_word, L.norm, L.rot);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool kRot, bool kNorm>
cudaError_t launch_any(const CUtensorMap &wmap, const CUtensorMap &xmap, const LinLaunch &L,
                       int B, int N, int K, const LinPlan &plan, uint32_t *error_word,
                       cudaStream_t stream) {
  const int splits = plan.splits;
  switch (plan.nb) {
    case 16:
      return launch_linear_nb<16, kRot, kNorm>(wmap, xmap, L, B, N, K, splits, error_word, stream);
    case 32:
      return launch_linear_nb<32, kRot, kNorm>(wmap, xmap, L, B, N, K, splits, error_word, stream);
    case 64:
      return launch_linear_nb<64, kRot, kNorm>(wmap, xmap, L, B, N, K, splits, error_word, stream);
    case 128:
      return launch_linear_nb<128, kRot, kNorm>(wmap, xmap, L, B, N, K, splits, error_word,
                                                stream);
    default:
      return launch_linear_nb<256, kRot, kNorm>(wmap, xmap, L, B, N, K, splits, error_word,
                                                stream);
  }
}

}  // namespace

int linear_batch_tile(int B) {
  return B <= 16 ? 16 : B <= 32 ? 32 : B <= 64 ? 64 : B <= 128 ? 128 : 256;
}

// The plan of a (B, N, K) projection on device `dev`: over the batch tiles that may
// serve B rows (the smallest that holds them; for more than 128 rows also 128, two or
// more tiles) and the K splits 1 .. 8 that leave no slice empty, the pair that
// minimises (waves of clusters) x (64-wide K pieces per CTA, weighted by the bytes a
// piece moves: 16 KB of weights plus nb x 128 bytes of activations, + a fixed cost for
// the CTA's start, pipeline fill and drain) + the cluster reduction, in units of a
// 32 KB piece's load time. A second wave is charged in full: its CTAs start only as
// the first ones leave.
LinPlan linear_plan(int B, int N, int K, int dev, bool norm, int forced_splits) {
  const int nb0 = linear_batch_tile(B);
  const int nsub = K / kLinSub;
  constexpr double kFixed = 8.0;
  LinPlan best{nb0, 1};
  double best_cost = 1e300;
  const int nbs[2] = {nb0, nb0 == 256 ? 128 : 0};
  for (int c = 0; c < 2; ++c) {
    const int nb = nbs[c];
    if (nb == 0) continue;
    const long long tiles = (long long)(N / kLinM) * ((B + nb - 1) / nb);
    // the tile choice is only weighed when it is open; otherwise both weights are 1.
    // A 256-row tile also has half again the fixed cost: its epilogue moves and
    // reduces a 128 KB accumulator (measured: 256 x 3072 x 2048 runs faster as two
    // 128-row tiles at K split 2, 256 x 6144 x 4096 as one 256-row tile at split 2).
    const double piece = nb0 == 256 ? (16384.0 + nb * 128.0) / 32768.0 : 1.0;
    const double fixed = nb == 256 ? 1.5 * kFixed : kFixed;
    for (int s = 1; s <= kMaxCluster && s <= nsub; ++s) {
      if (forced_splits > 0 && s != forced_splits) continue;
      const int cps = (nsub + s - 1) / s;
      if ((nsub + cps - 1) / cps != s) continue;  // that split would leave a slice empty
      const int res = norm ? resident<true>(nb, dev, s) : resident<false>(nb, dev, s);
      if (res <= 0) continue;
      const long long waves = (tiles + res - 1) / res;
      const double reduce = s > 1 ? (double)nb * (s - 1) / (50.0 * s) : 0.0;
      const double cost = (double)waves * (cps * piece + fixed) + reduce;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = LinPlan{nb, s};
      }
    }
  }
  if (best_cost == 1e300 && forced_splits > 0) best.splits = forced_splits;
  // a forced split that would leave a slice empty becomes the even one
  const int cps = (nsub + best.splits - 1) / best.splits;
  best.splits = (nsub + cps - 1) / cps;
  return best;
}

cudaError_t launch_linear(const CUtensorMap &wmap, const CUtensorMap &xmap, const void *residual,
                          void *y, int B, int N, int K, const LinPlan &plan,
                          uint32_t *error_word, cudaStream_t stream) {
  LinLaunch L{};
  L.rmap = &xmap;
  L.residual = residual;
  L.y = y;
  return launch_any<false, false>(wmap, xmap, L, B, N, K, plan, error_word, stream);
}

cudaError_t launch_linear_norm(const CUtensorMap &wmap, const CUtensorMap &xmap,
                               const CUtensorMap &rmap, const LinNorm &norm, void *y, int B,
                               int N, int K, const LinPlan &plan, uint32_t *error_word,
                               cudaStream_t stream) {
  LinLaunch L{};
  L.rmap = &rmap;
  L.y = y;
  L.norm = norm;
  return launch_any<false, true>(wmap, xmap, L, B, N, K, plan, error_word, stream);
}

cudaError_t launch_linear_qkv_rot(const CUtensorMap &wmap, const CUtensorMap &xmap, int B,
                                  int N, int K, const LinPlan &plan, const QkvRotArgs &rot,
                                  uint32_t *error_word, cudaStream_t stream,
                                  const CUtensorMap *rmap, const LinNorm *norm) {
  LinLaunch L{};
  L.rot = rot;
  if (norm != nullptr) {
    L.rmap = rmap != nullptr ? rmap : &xmap;
    L.norm = *norm;
    return launch_any<true, true>(wmap, xmap, L, B, N, K, plan, error_word, stream);
  }
  L.rmap = &xmap;
  return launch_any<true, false>(wmap, xmap, L, B, N, K, plan, error_word, stream);
}

}  // namespace decattn
