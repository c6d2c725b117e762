// K3 + K4: single-query GQA decode attention over a contiguous bf16 KV cache.
//
// fusedtok README, "Operators" (attention_decode: single-token causal attention
// with GQA over a contiguous kv-cache, online softmax, flash-decoding split over
// long caches, per-sequence lengths) and "Usage" (q [B,Hq,D], caches [B,Hkv,T,D],
// lens [B] int32); "Benchmarks" (one launch streams the GQA cache once; heads are
// expanded with repeat_interleave, so query head h reads KV head h / G).
//
// Split pass (K3). The Hkv * sum(lens) rows (sequence b, KV head g, token t) are read
// as one stream, ordered by (b, g, t), and cut into gridDim.x equal contiguous pieces;
// CTA c owns rows [c*per, (c+1)*per). Every CTA therefore streams the same number of
// K/V bytes whatever the length mix, and a piece that crosses a (b, g) boundary
// produces one partial per pair it touches, stored in slot c + b*Hkv + g (distinct
// for every touching (c, pair), since pieces and pairs are both contiguous).
//
// Inside a CTA one producer lane issues 128B-swizzled bulk-tensor (TMA) loads of
// 64-token K and V tiles into a 4-stage shared-memory ring guarded by mbarriers.
// Eight consumer warps in two groups take alternate tiles; a warp owns 16 token rows
// of a tile and serves all G <= 8 query heads of the KV head from that one read:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T        (mma m16n8k16, bf16 -> fp32)
//   online softmax per head column (base-2 exponent, running max and sum)
//   O^T[D x 8 heads]     += V^T[D x 16] . P^T      (P split into bf16 hi + lo parts,
//                                                   two mma, ~16-bit weights)
// The S^T accumulator layout turns into the P^T operand layout with one 8x8
// register transpose (movmatrix), so P never touches shared memory. At the end of a
// pair the warps' (m, l, O) are combined through shared memory and the partial
// (normalised o and lse, base 2) is written.
//
// Merge pass (K4). One CTA per sequence, one warp per query head: walk the partials
// of the head's (b, g) pair in order with a running log-sum-exp and write bf16 out.
#include <math.h>

#include "dec_device.cuh"
#include "dec_launch.h"

namespace decattn {
namespace {

constexpr int kTile = kSplitTile;       // tokens per stage
constexpr int kGroupWarps = 4;          // 4 warps x 16 rows = one tile
constexpr int kGroups = 2;              // tiles alternate between warp groups
constexpr int kConsumerWarps = kGroupWarps * kGroups;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kStages = 4;
constexpr int kMaxG = 8;

template <int D>
struct Geom {
  static constexpr int kBoxes = D / 64;             // 128-byte swizzle boxes per row
  static constexpr int kBoxBytes = kTile * 128;     // one box of one tile
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
  static constexpr int kOStride = D + 4;            // floats between heads in the combine area
  static constexpr int kWarpScratch = kMaxG * kOStride + 2 * kMaxG;  // floats per warp
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kScratchOffset = kBarOffset + 2 * kStages * 8;
  static constexpr int kPrefixOffset = kScratchOffset + kConsumerWarps * kWarpScratch * 4;
  static size_t smem_bytes(int B) { return 1024 + kPrefixOffset + (size_t)(B + 1) * 4 + 16; }
};

// A run of one (b, g) pair's tokens [t0, t1) inside this CTA's piece.
struct Seg {
  int b, g, t0, t1;
  long long r;   // stream row of t0
};

__device__ __forceinline__ int seq_len(const int *prefix, int b) { return prefix[b + 1] - prefix[b]; }

__device__ __forceinline__ Seg first_seg(const int *prefix, int B, int Hkv, long long r0,
                                         long long r1) {
  // the last sequence whose first row is <= r0 (it is non-empty since r0 < total)
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)Hkv * prefix[mid] <= r0) lo = mid; else hi = mid - 1;
  }
  Seg s;
  s.b = lo;
  const int L = seq_len(prefix, lo);
  const long long within = r0 - (long long)Hkv * prefix[lo];
  s.g = (int)(within / L);
  s.t0 = (int)(within % L);
  s.t1 = (int)min((long long)L, (long long)s.t0 + (r1 - r0));
  s.r = r0;
  return s;
}

__device__ __forceinline__ bool next_seg(const int *prefix, int Hkv, long long r1, Seg &s) {
  s.r += s.t1 - s.t0;
  if (s.r >= r1) return false;
  if (++s.g == Hkv) {
    s.g = 0;
    do { ++s.b; } while (seq_len(prefix, s.b) == 0);
  }
  s.t0 = 0;
  s.t1 = (int)min((long long)seq_len(prefix, s.b), r1 - s.r);
  return true;
}

__device__ __forceinline__ void named_bar_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Shared address of (row, 16-byte chunk) of a tile written by a SWIZZLE_128B TMA box:
// chunk c of row r lands at chunk c ^ (r & 7) of that row's 128 bytes.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * Geom<D>::kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) gqa_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ lens, int B, int Hq,
    int Hkv, int T_cap, float scale_log2, uint8_t *__restrict__ workspace) {
  using Gm = Geom<D>;
  constexpr int KS = D / 16;  // k-steps of S^T = K Q^T
  constexpr int MT = D / 16;  // m-tiles of O^T = V^T P^T
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_warp_tot[kThreads / 32];
  __shared__ volatile int s_abort;

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar_full = s_base + Gm::kBarOffset;            // kStages x 8 bytes
  const uint32_t bar_empty = bar_full + kStages * 8;
  float *scratch = reinterpret_cast<float *>(smem + Gm::kScratchOffset);
  int *prefix = reinterpret_cast<int *>(smem + Gm::kPrefixOffset);
  uint32_t *err = reinterpret_cast<uint32_t *>(workspace);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = Hq / Hkv;

  // ---- prologue: clamped lengths -> exclusive prefix sums in shared memory
  {
    const int chunk = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * chunk), b1 = min(B, b0 + chunk);
    int local = 0;
    bool clamped = false;
    for (int b = b0; b < b1; ++b) {
      int L = lens[b];
      if (L < 0 || L > T_cap) { clamped = true; L = L < 0 ? 0 : T_cap; }
      local += L;
    }
    if (clamped) atomicOr(err, kErrLenClamped);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp_tot[warp] = incl;
    if (tid == 0) s_abort = 0;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp_tot[w];
    int run = before + incl - local;
    for (int b = b0; b < b1; ++b) {
      prefix[b] = run;
      int L = lens[b];
      L = L < 0 ? 0 : (L > T_cap ? T_cap : L);
      run += L;
    }
    if (tid == kThreads - 1) prefix[B] = before + incl;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kGroupWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const long long total = (long long)Hkv * prefix[B];
  const long long per = rows_per_part(total, gridDim.x);
  const long long r0 = (long long)blockIdx.x * per;
  if (r0 >= total) return;  // uniform over the CTA; nothing was issued yet
  const long long r1 = min(r0 + per, total);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      const uint64_t policy = l2_policy_evict_first();
      int it = 0;
      int last_n[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_n[s] = -1;
      Seg sg = first_seg(prefix, B, Hkv, r0, r1);
      do {
        const int pair = sg.b * Hkv + sg.g;
        for (int tt = sg.t0; tt < sg.t1; tt += kTile, ++it) {
          const int st = it % kStages, n = it / kStages;
          if (s_abort) continue;
          if (n > 0 && !mbar_wait_bounded(bar_empty + 8 * st, (n - 1) & 1)) {
            atomicOr(err, kErrWaitTimeout);
            s_abort = 1;
            continue;
          }
          const uint32_t full = bar_full + 8 * st;
          mbar_arrive_expect_tx(full, Gm::kStageBytes);
          const uint32_t kt = s_base + st * Gm::kStageBytes;
          const uint32_t vt = kt + Gm::kTileBytes;
#pragma unroll
          for (int bx = 0; bx < Gm::kBoxes; ++bx) {
            tma_load_3d(kt + bx * Gm::kBoxBytes, &kmap, bx * 64, tt, pair, full, policy);
            tma_load_3d(vt + bx * Gm::kBoxBytes, &vmap, bx * 64, tt, pair, full, policy);
          }
          last_n[st] = n;
        }
      } while (next_seg(prefix, Hkv, r1, sg));
      // no copy may still be in flight into this CTA's shared memory when it exits
#pragma unroll
      for (int s = 0; s < kStages; ++s)
        if (last_n[s] >= 0) mbar_wait_bounded(bar_full + 8 * s, last_n[s] & 1);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int grp = warp / kGroupWarps;
  const int row0 = 16 * (warp % kGroupWarps);  // first tile row of this warp
  const int gid = lane >> 2, tig = lane & 3;
  const float NEG_INF = -INFINITY;
  float *o_ws = reinterpret_cast<float *>(workspace + kWorkspaceHeaderBytes);
  const size_t slots = (size_t)gridDim.x + (size_t)B * Hkv;
  float *lse_ws = o_ws + slots * G * D;

  int it = 0;
  Seg sg = first_seg(prefix, B, Hkv, r0, r1);
  do {
    const int pair = sg.b * Hkv + sg.g;
    const int L = seq_len(prefix, sg.b);
    // Q^T operand (k = head dim, n = query head of the group); heads >= G are zero.
    uint32_t qf[KS][2];
    {
      const bool hv = gid < G;
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          q + ((size_t)sg.b * Hq + (size_t)sg.g * G + (hv ? gid : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][0] = hv ? __ldg(qrow + (16 * ks + 2 * tig) / 2) : 0u;
        qf[ks][1] = hv ? __ldg(qrow + (16 * ks + 8 + 2 * tig) / 2) : 0u;
      }
    }
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int tt = sg.t0; tt < sg.t1; tt += kTile, ++it) {
      if (it % kGroups != grp) continue;
      const int st = it % kStages, n = it / kStages;
      if (!s_abort && !mbar_wait_bounded(bar_full + 8 * st, n & 1)) {
        if (lane == 0) atomicOr(err, kErrWaitTimeout);
        s_abort = 1;
      }
      const int tok0 = tt + row0;  // token of this warp's first row
      if (!s_abort && tok0 < sg.t1) {
        const uint32_t kt = s_base + st * Gm::kStageBytes;
        const uint32_t vt = kt + Gm::kTileBytes;
        if (tok0 + 16 > L) {
          // rows at or past the sequence length hold no data (possibly NaN): zero their V
          const int rlo = max(L - tt, row0);
          const int nrows = row0 + 16 - rlo;
          uint8_t *vtile = smem + st * Gm::kStageBytes + Gm::kTileBytes;
          for (int i = lane; i < nrows * Gm::kBoxes * 8; i += 32) {
            const int r = rlo + i / (Gm::kBoxes * 8);
            const int rest = i % (Gm::kBoxes * 8);
            *reinterpret_cast<uint4 *>(vtile + (rest >> 3) * Gm::kBoxBytes + r * 128 +
                                       (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        // ---- S^T = K . Q^T over this warp's 16 rows (two accumulators for ILP)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int r = row0 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int csel = lane >> 4;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(tile_addr<D>(kt, r, 2 * ks + csel), a[0], a[1], a[2], a[3]);
            if (ks & 1) mma_bf16_16816(sb, a, qf[ks][0], qf[ks][1]);
            else mma_bf16_16816(sa, a, qf[ks][0], qf[ks][1]);
          }
        }
        // ---- online softmax; this lane holds tokens (gid, gid+8) x heads (2tig, 2tig+1)
        const bool va = tok0 + gid < sg.t1, vb = tok0 + gid + 8 < sg.t1;
        const float x0 = va ? (sa[0] + sb[0]) * scale_log2 : NEG_INF;
        const float x1 = va ? (sa[1] + sb[1]) * scale_log2 : NEG_INF;
        const float x2 = vb ? (sa[2] + sb[2]) * scale_log2 : NEG_INF;
        const float x3 = vb ? (sa[3] + sb[3]) * scale_log2 : NEG_INF;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
        const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
          }
        }
        // ---- P^T operand: hi = bf16(p), lo = bf16(p - hi); transpose 8x8 blocks
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        const uint32_t e01 = pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        const uint32_t e23 = pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
        const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
        const uint32_t bl0 = movmatrix_trans(e01), bl1 = movmatrix_trans(e23);
        // ---- O^T += V^T . P^T
        {
          const int r = row0 + (lane & 7) + 8 * (lane >> 4);
          const int csel = (lane >> 3) & 1;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(tile_addr<D>(vt, r, 2 * mt + csel), a[0], a[1], a[2], a[3]);
            mma_bf16_16816(o[mt], a, bh0, bh1);
            mma_bf16_16816(o[mt], a, bl0, bl1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }

    // ---- combine the warps' states of this pair into one partial
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    {
      float *sw = scratch + warp * Gm::kWarpScratch;
      float *sm = sw + kMaxG * Gm::kOStride;
      float *sl = sm + kMaxG;
      const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int d = 16 * mt + gid;
        sw[h0 * Gm::kOStride + d] = o[mt][0];
        sw[h1 * Gm::kOStride + d] = o[mt][1];
        sw[h0 * Gm::kOStride + d + 8] = o[mt][2];
        sw[h1 * Gm::kOStride + d + 8] = o[mt][3];
      }
      if (gid == 0) {
        sm[h0] = m0; sl[h0] = l0;
        sm[h1] = m1; sl[h1] = l1;
      }
    }
    named_bar_consumers();
    {
      const size_t slot = (size_t)blockIdx.x + pair;
      float *op = o_ws + slot * G * D;
      for (int e = tid; e < G * D; e += kConsumerThreads) {
        const int h = e / D, d = e - h * D;
        float M = NEG_INF;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
          M = fmaxf(M, scratch[w * Gm::kWarpScratch + kMaxG * Gm::kOStride + h]);
        float wsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float *sw = scratch + w * Gm::kWarpScratch;
          const float mw = sw[kMaxG * Gm::kOStride + h];
          const float f = (mw == NEG_INF) ? 0.f : exp2f(mw - M);
          wsum += f * sw[kMaxG * Gm::kOStride + kMaxG + h];
          acc += f * sw[h * Gm::kOStride + d];
        }
        op[e] = acc / wsum;
        if (d == 0) lse_ws[slot * G + h] = M + log2f(wsum);
      }
    }
    named_bar_consumers();
  } while (next_seg(prefix, Hkv, r1, sg));
}

template <int D>
__global__ void __launch_bounds__(256) split_merge_kernel(const uint8_t *__restrict__ workspace,
                                                          const int32_t *__restrict__ lens,
                                                          __nv_bfloat16 *__restrict__ out, int B,
                                                          int Hq, int Hkv, int T_cap,
                                                          int num_parts) {
  constexpr int E = D / 32;  // floats per lane
  __shared__ int s_red[2][8];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = Hq / Hkv;
  // total rows and the rows before sequence b (lengths clamped as in the split pass)
  int tot = 0, pre = 0;
  for (int i = tid; i < B; i += 256) {
    int L = lens[i];
    L = L < 0 ? 0 : (L > T_cap ? T_cap : L);
    tot += L;
    if (i < b) pre += L;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
  }
  if (lane == 0) { s_red[0][warp] = tot; s_red[1][warp] = pre; }
  __syncthreads();
  tot = 0; pre = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) { tot += s_red[0][w]; pre += s_red[1][w]; }
  int Lb = lens[b];
  Lb = Lb < 0 ? 0 : (Lb > T_cap ? T_cap : Lb);
  const long long per = rows_per_part((long long)Hkv * tot, num_parts);
  const float *o_ws = reinterpret_cast<const float *>(workspace + kWorkspaceHeaderBytes);
  const size_t slots = (size_t)num_parts + (size_t)B * Hkv;
  const float *lse_ws = o_ws + slots * G * D;

  for (int h = warp; h < Hq; h += 8) {
    __nv_bfloat16 *orow = out + ((size_t)b * Hq + h) * D + lane * E;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float wsum = 1.f;
    if (Lb > 0) {
      const int g = h / G, hh = h - g * G;
      const int pair = b * Hkv + g;
      const long long start = (long long)Hkv * pre + (long long)g * Lb;
      const long long c0 = start / per, c1 = (start + Lb - 1) / per;
      float M = -INFINITY;
      wsum = 0.f;
      for (long long c = c0; c <= c1; ++c) {
        const size_t slot = (size_t)c + pair;
        const float lse = lse_ws[slot * G + hh];
        if (lse > M) {
          const float sc = exp2f(M - lse);
          wsum *= sc;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] *= sc;
          M = lse;
        }
        const float w = exp2f(lse - M);
        wsum += w;
        const float *op = o_ws + (slot * G + hh) * D + lane * E;
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4 *>(op);
          acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2 *>(op);
          acc[0] += w * v.x; acc[1] += w * v.y;
        }
      }
    }
    const float inv = 1.f / wsum;
    if constexpr (E == 4) {
      *reinterpret_cast<uint2 *>(orow) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                    pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
      *reinterpret_cast<uint32_t *>(orow) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
  }
}

template <int D>
cudaError_t ensure_split_attr(int device) {
  static int done[64] = {0};
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gqa_split_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Geom<D>::smem_bytes(kSplitMaxB));
  if (e == cudaSuccess) done[device] = 1;
  return e;
}

}  // namespace

size_t split_smem_bytes(int D, int B) {
  return D == 128 ? Geom<128>::smem_bytes(B) : Geom<64>::smem_bytes(B);
}

int split_ctas_per_sm(int D, int B, int device) {
  int n = 0;
  const size_t smem = split_smem_bytes(D, B);
  cudaError_t e;
  if (D == 128) {
    if (ensure_split_attr<128>(device) != cudaSuccess) return 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_split_kernel<128>, kThreads, smem);
  } else {
    if (ensure_split_attr<64>(device) != cudaSuccess) return 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_split_kernel<64>, kThreads, smem);
  }
  if (e != cudaSuccess || n < 1) return 1;
  return n;
}

cudaError_t launch_gqa_split(const CUtensorMap &kmap, const CUtensorMap &vmap, const void *q,
                             const int32_t *lens, int B, int Hq, int Hkv, int D, int T_cap,
                             float scale_log2, int num_parts, void *workspace,
                             cudaStream_t stream) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const size_t smem = split_smem_bytes(D, B);
  auto *qp = static_cast<const __nv_bfloat16 *>(q);
  auto *ws = static_cast<uint8_t *>(workspace);
  if (D == 128) {
    if ((e = ensure_split_attr<128>(device)) != cudaSuccess) return e;
    gqa_split_kernel<128><<<num_parts, kThreads, smem, stream>>>(kmap, vmap, qp, lens, B, Hq, Hkv,
                                                                 T_cap, scale_log2, ws);
  } else {
    if ((e = ensure_split_attr<64>(device)) != cudaSuccess) return e;
    gqa_split_kernel<64><<<num_parts, kThreads, smem, stream>>>(kmap, vmap, qp, lens, B, Hq, Hkv,
                                                                T_cap, scale_log2, ws);
  }
  return cudaGetLastError();
}

cudaError_t launch_split_merge(const void *workspace, const int32_t *lens, void *out, int B,
                               int Hq, int Hkv, int D, int T_cap, int num_parts,
                               cudaStream_t stream) {
  auto *ws = static_cast<const uint8_t *>(workspace);
  auto *op = static_cast<__nv_bfloat16 *>(out);
  if (D == 128)
    split_merge_kernel<128><<<B, 256, 0, stream>>>(ws, lens, op, B, Hq, Hkv, T_cap, num_parts);
  else
    split_merge_kernel<64><<<B, 256, 0, stream>>>(ws, lens, op, B, Hq, Hkv, T_cap, num_parts);
  return cudaGetLastError();
}

}  // namespace decattn
