// The sampling side of a decode step, fused into one launch (fusedtok 1.0.1 README,
// "Operators": repetition penalty, temperature, argmax, sample_topk, sample_topp,
// decode_step = penalty -> temperature -> nucleus sample; "Usage": one call per step).
//
// One thread-block cluster of C CTAs per row of logits (C a power of two, up to 16): CTA r keeps
// slice r of the row in shared memory, every pass after the load runs out of shared
// memory, and the CTAs combine their partial results through distributed shared
// memory. Per row:
//   1. load the slice; apply the CTRL penalty to the listed ids (each writer computes
//      the penalised value from the original logit, so repeated ids apply once);
//   2. temperature <= 0: argmax (ties to the lowest id) and stop; else z / T, the row
//      maximum, e = exp(z - max);
//   3. probability masses as 64-bit fixed point, m = round(e * 2^40): every sum below is
//      an integer sum, exact and independent of order;
//   4. top-k: a radix select over the bit patterns of e (4 passes of 8 bits, per-bucket
//      counts; when the first pass leaves at most 2048 members in the chosen bucket, the
//      other three run on one CTA over those members) finds the k-th largest value;
//      equal values are ranked by token id;
//   5. top-p: the same radix select over the top-k survivors with per-bucket masses
//      finds the last member of the shortest prefix of the ranking whose mass reaches
//      p times the survivors' mass;
//   6. the draw: target = floor(u * nucleus mass); the token is the first member, in
//      token-id order, whose running mass exceeds it (a scan over threads and CTAs).
// Each thread owns a contiguous chunk of its CTA's slice, so every scan in token-id
// order is a sequential walk inside a chunk plus exclusive sums over threads and CTAs.
// The slice is stored with one padding word per 32 values so that the threads' chunks
// fall on different shared-memory banks.
#include <cuda_runtime.h>

#include <atomic>
#include <math.h>

#include "dec_device.cuh"
#include "dec_launch.h"

namespace decattn {
namespace {

constexpr int kSmpThreads = 512;
constexpr int kSmpWarps = kSmpThreads / 32;
constexpr int kBuckets = 256;
constexpr uint32_t kMaxCl = 16;  // largest cluster (CTAs per row)
// Radix-select histograms: one per group of kSmpWarps / G warps. A mass is added as two
// 32-bit parts (its low 20 bits and the rest), which stays exact while a group sees at
// most 2^12 elements per pass: a slice of at most G * 2^12 (half that is allowed, for
// margin). Two builds of the kernel: G = 16 (a histogram per warp, no contention) for a
// few rows, each cluster on SMs of its own; G = 8 for batches, small enough in shared
// memory and registers for two CTAs per SM.
constexpr int kLatencyGroups = 16;
constexpr int kBatchGroups = 8;
__host__ __device__ constexpr int max_slice(int G) { return G * 4096 / 2; }
// Candidates of the chosen top-byte bucket kept for the later radix passes; a bucket
// with more members (a flat row) is found again by walking the slice.
constexpr int kCandCap = 2048;

struct SmpArgs {
  const float *logits;
  const int32_t *ids;
  const float *u;
  int32_t *tokens;
  int V, L, slice;
  float penalty, temperature, top_p;
  int top_k;
};

__device__ __forceinline__ int padded(int i) { return i + (i >> 5); }

// One warp group's histogram of a radix pass.
struct WarpHist {
  unsigned int cnt[kBuckets];
  unsigned int lo[kBuckets];  // sums of the low 20 bits of the masses
  unsigned int hi[kBuckets];  // sums of the masses shifted right by 20
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t map_rank(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t ld_cl_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_cl_u64(uint32_t a) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float ld_cl_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// Shared state of one CTA. `pub_*` are written by this CTA and read by the others of
// the cluster after a cluster barrier; they alternate between two slots so that a CTA
// never overwrites a slot a peer may still be reading.
struct SmpShared {
  unsigned int pub_cnt[2][kBuckets];
  unsigned long long pub_mass[2][kBuckets];
  float pub_f[2];
  int pub_i[2];
  unsigned long long pub_u64[2][2];
  unsigned int pub_n[2];                 // this CTA's candidate count
  unsigned long long pub_sel[2][3];      // CTA 0's selection: tau, above, eq_cnt
  unsigned int cnt[kBuckets];  // this CTA's histogram, then the cluster's
  unsigned long long mass[kBuckets];
  unsigned long long warp_u64[kSmpWarps][2];
  float warp_f[kSmpWarps];
  int warp_i[kSmpWarps];
  unsigned long long bc_u64[4];
  unsigned int bc_u32[4];
  float bc_f;
  int bc_i;
};

// round(e * 2^40) for e in [0, 1], from the bits of e with integer shifts: e =
// mant * 2^(ex - 150) with the 24-bit significand mant, so e * 2^40 = mant * 2^(ex - 110).
__device__ __forceinline__ unsigned long long to_mass(float e) {
  const uint32_t bits = __float_as_uint(e);
  const int ex = (int)(bits >> 23);
  if (ex == 0) return 0;  // zero or subnormal: below 2^-126, far under one unit
  const unsigned long long mant = (bits & 0x7FFFFFu) | 0x800000u;
  const int sh = ex - 110;
  if (sh >= 0) return mant << sh;
  if (sh < -24) return 0;
  return (mant + (1ull << (-sh - 1))) >> (-sh);
}

// Block-wide exclusive prefix (in thread order) of a 64-bit value; `total` gets the sum.
__device__ unsigned long long block_exclusive_u64(unsigned long long v, SmpShared &sh,
                                                  unsigned long long &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh.warp_u64[warp][0] = incl;
  __syncthreads();
  unsigned long long before = 0;
  total = 0;
  for (int w = 0; w < kSmpWarps; ++w) {
    if (w < warp) before += sh.warp_u64[w][0];
    total += sh.warp_u64[w][0];
  }
  __syncthreads();
  return before + incl - v;
}

// Cluster-wide exclusive prefix (in CTA rank order) of one per-CTA 64-bit value.
__device__ unsigned long long cluster_exclusive_u64(unsigned long long mine, SmpShared &sh,
                                                    int &slot, unsigned long long &total) {
  const uint32_t C = gridDim.x, rank = cluster_rank();
  if (threadIdx.x == 0) sh.pub_u64[slot][0] = mine;
  cluster_sync_all();
  if (threadIdx.x == 0) {
    unsigned long long v[kMaxCl];
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < C) v[q] = ld_cl_u64(map_rank(&sh.pub_u64[slot][0], q));
    unsigned long long before = 0, all = 0;
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < C) {
        if (q < rank) before += v[q];
        all += v[q];
      }
    sh.bc_u64[0] = before;
    sh.bc_u64[1] = all;
  }
  __syncthreads();
  total = sh.bc_u64[1];
  const unsigned long long r = sh.bc_u64[0];
  __syncthreads();
  slot ^= 1;
  return r;
}

// The cluster-wide maximum of one float per thread.
__device__ float cluster_max(float v, SmpShared &sh, int &slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sh.warp_f[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = sh.warp_f[0];
    for (int w = 1; w < kSmpWarps; ++w) m = fmaxf(m, sh.warp_f[w]);
    sh.pub_f[slot] = m;
  }
  cluster_sync_all();
  if (threadIdx.x == 0) {
    float v[kMaxCl];
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < gridDim.x) v[q] = ld_cl_f32(map_rank(&sh.pub_f[slot], q));
    float m = -INFINITY;
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < gridDim.x) m = fmaxf(m, v[q]);
    sh.bc_f = m;
  }
  __syncthreads();
  const float r = sh.bc_f;
  __syncthreads();
  slot ^= 1;
  return r;
}

// Cluster-wide argmax of (value, index): the largest value, the lowest index among equals.
__device__ int cluster_argmax(float v, int idx, SmpShared &sh, int &slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > v || (ov == v && oi < idx)) {
      v = ov;
      idx = oi;
    }
  }
  if (lane == 0) {
    sh.warp_f[warp] = v;
    sh.warp_i[warp] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv = sh.warp_f[0];
    int bi = sh.warp_i[0];
    for (int w = 1; w < kSmpWarps; ++w)
      if (sh.warp_f[w] > bv || (sh.warp_f[w] == bv && sh.warp_i[w] < bi)) {
        bv = sh.warp_f[w];
        bi = sh.warp_i[w];
      }
    sh.pub_f[slot] = bv;
    sh.pub_i[slot] = bi;
  }
  cluster_sync_all();
  if (threadIdx.x == 0) {
    float fv[kMaxCl];
    int iv[kMaxCl];
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < gridDim.x) {
        fv[q] = ld_cl_f32(map_rank(&sh.pub_f[slot], q));
        iv[q] = (int)ld_cl_u32(map_rank(&sh.pub_i[slot], q));
      }
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < gridDim.x && (fv[q] > bv || (fv[q] == bv && iv[q] < bi))) {
        bv = fv[q];
        bi = iv[q];
      }
    sh.bc_i = bi;
  }
  __syncthreads();
  const int r = sh.bc_i;
  __syncthreads();
  slot ^= 1;
  return r;
}

// Membership of the elements of one chunk, walked in token-id order: the top-k set
// (key above tauK, or equal to it and among the first needK equal ones by id) and,
// within it, the nucleus (same rule with tauP / needP). eq*_start are the numbers of
// equal elements before this chunk in token-id order.
struct Member {
  bool use_k, use_p;
  uint32_t tau_k, tau_p;
  unsigned long long need_k, need_p;
};

// Radix-select histograms, one per warp group (kWarpsPerHist warps share one, so the
// CTA's histograms stay small enough for two CTAs per SM). A mass is added as two
// 32-bit parts, its low 20 bits and the rest, so every sum stays an exact integer sum
// (a group sees at most 2^12 elements per pass). When the 32 lanes of a step all hit
// the same bucket (flat rows, later passes), one lane adds the warp's sums.
__device__ __forceinline__ void hist_add(WarpHist &h, int b, unsigned long long m) {
  const int lane = threadIdx.x & 31;
  const unsigned lo = (unsigned)(m & 0xFFFFFull), hi = (unsigned)(m >> 20);
  const int b_first = __shfl_sync(0xffffffffu, b, 0);
  if (__all_sync(0xffffffffu, b == b_first)) {
    if (b_first < kBuckets) {
      const unsigned slo = __reduce_add_sync(0xffffffffu, lo);
      const unsigned shi = __reduce_add_sync(0xffffffffu, hi);
      if (lane == 0) {
        atomicAdd(&h.cnt[b_first], 32u);
        atomicAdd(&h.lo[b_first], slo);
        atomicAdd(&h.hi[b_first], shi);
      }
    }
  } else if (b < kBuckets) {
    atomicAdd(&h.cnt[b], 1u);
    atomicAdd(&h.lo[b], lo);
    atomicAdd(&h.hi[b], hi);
  }
  __syncwarp();
}

// Clears every group's histogram before the first add of a pass. With a histogram per
// warp each warp clears its own; shared ones are cleared by the CTA, then a barrier.
// (The previous pass's reads of every histogram finished before its cluster barrier.)
template <int G>
__device__ __forceinline__ void hist_clear(WarpHist *wh) {
  if constexpr (G == kSmpWarps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = lane; b < kBuckets; b += 32) {
      wh[warp].cnt[b] = 0;
      wh[warp].lo[b] = 0;
      wh[warp].hi[b] = 0;
    }
    __syncwarp();
  } else {
    for (int i = threadIdx.x; i < G * kBuckets; i += kSmpThreads) {
      const int g = i / kBuckets, b = i - g * kBuckets;
      wh[g].cnt[b] = 0;
      wh[g].lo[b] = 0;
      wh[g].hi[b] = 0;
    }
    __syncthreads();
  }
}

// Sum the groups' histograms, publish this CTA's, and leave the cluster's histogram
// (the sum over CTAs, in rank order) in sh.cnt / sh.mass.
template <int G>
__device__ void hist_merge(WarpHist *wh, SmpShared &sh, int &slot) {
  __syncthreads();
  for (int b = threadIdx.x; b < kBuckets; b += kSmpThreads) {
    unsigned int c = 0;
    unsigned long long ms = 0;
    for (int w = 0; w < G; ++w) {
      c += wh[w].cnt[b];
      ms += (unsigned long long)wh[w].lo[b] + ((unsigned long long)wh[w].hi[b] << 20);
    }
    sh.pub_cnt[slot][b] = c;
    sh.pub_mass[slot][b] = ms;
  }
  cluster_sync_all();
  for (int b = threadIdx.x; b < kBuckets; b += kSmpThreads) {
    unsigned int cv[kMaxCl];
    unsigned long long mv[kMaxCl];
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < gridDim.x) {
        cv[q] = ld_cl_u32(map_rank(&sh.pub_cnt[slot][b], q));
        mv[q] = ld_cl_u64(map_rank(&sh.pub_mass[slot][b], q));
      }
    unsigned int c = 0;
    unsigned long long ms = 0;
#pragma unroll
    for (uint32_t q = 0; q < kMaxCl; ++q)
      if (q < gridDim.x) {
        c += cv[q];
        ms += mv[q];
      }
    sh.cnt[b] = c;
    sh.mass[b] = ms;
  }
  __syncthreads();
  slot ^= 1;
}

// Find the bucket where the running total from the top (count when by_mass is false,
// else mass), started at `above`, first reaches `target`; returns it and adds the
// total of the buckets above it to `above`. Also reports that bucket's count and mass.
__device__ int radix_pick(bool by_mass, unsigned long long target, unsigned long long &above,
                          unsigned int &bucket_cnt, unsigned long long &bucket_mass,
                          SmpShared &sh) {
  // suffix sums from bucket 255 down, computed by one warp (8 buckets per lane)
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long local[8];
    unsigned long long acc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // lane 0 holds buckets 255..248, lane 1 247..240, ...
      const int b = 255 - (lane * 8 + j);
      acc += by_mass ? sh.mass[b] : (unsigned long long)sh.cnt[b];
      local[j] = acc;
    }
    unsigned long long incl = acc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const unsigned long long before_lane = incl - acc;
    int found = -1;
    unsigned long long found_above = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const unsigned long long upto = above + before_lane + local[j];
      const unsigned long long prev = above + before_lane + (j ? local[j - 1] : 0ull);
      if (found < 0 && upto >= target && prev < target) {
        found = 255 - (lane * 8 + j);
        found_above = prev;
      }
    }
    // the first lane (highest buckets) that found a crossing wins; if the target is
    // beyond the total (rounding), take the lowest non-empty bucket
    const unsigned int ballot = __ballot_sync(0xffffffffu, found >= 0);
    if (ballot != 0) {
      const int src = __ffs(ballot) - 1;
      if (lane == src) {
        sh.bc_u32[0] = (unsigned)found;
        sh.bc_u64[2] = found_above;
      }
    } else if (lane == 0) {
      int b = 0;
      unsigned long long tot = 0;
      for (int k = 255; k >= 0; --k) {
        const unsigned long long w = by_mass ? sh.mass[k] : (unsigned long long)sh.cnt[k];
        if (w) b = k;
      }
      for (int k = 255; k > b; --k) tot += by_mass ? sh.mass[k] : (unsigned long long)sh.cnt[k];
      sh.bc_u32[0] = (unsigned)b;
      sh.bc_u64[2] = above + tot;
    }
  }
  __syncthreads();
  const int b = (int)sh.bc_u32[0];
  above = sh.bc_u64[2];
  bucket_cnt = sh.cnt[b];
  bucket_mass = sh.mass[b];
  __syncthreads();
  return b;
}

// Walker over a chunk in token-id order deciding top-k membership.
struct InK {
  const Member *m;
  unsigned long long eq_start, eq_seen;
  __device__ void begin() { eq_seen = eq_start; }
  __device__ bool next(uint32_t key) {
    if (!m->use_k) return true;
    if (key > m->tau_k) return true;
    if (key == m->tau_k) return eq_seen++ < m->need_k;
    return false;
  }
};

// Walker deciding nucleus membership (top-k, then top-p).
struct InNucleus {
  InK k;
  const Member *m;
  unsigned long long eq_start, eq_seen;
  __device__ void begin() {
    k.begin();
    eq_seen = eq_start;
  }
  __device__ bool next(uint32_t key) {
    if (!k.next(key)) return false;
    if (!m->use_p) return true;
    if (key > m->tau_p) return true;
    if (key == m->tau_p) return eq_seen++ < m->need_p;
    return false;
  }
};

// Number of elements of the chunk with key == tau among the members of `set`.
template <typename Pred>
__device__ unsigned long long count_equal(const float *vals, int c0, int c1, uint32_t tau,
                                          Pred set) {
  unsigned long long n = 0;
  set.begin();
  for (int i = c0; i < c1; ++i) {
    const uint32_t key = __float_as_uint(vals[padded(i)]);
    if (set.next(key) && key == tau) ++n;
  }
  return n;
}

// The rest of a radix select once every CTA has gathered its candidates (at most
// kCandCap over the cluster) into `cand`: CTA 0 collects the cluster's candidates into
// `buf` (distributed shared memory) and runs the 8-bit passes first_pass .. 3 over them
// alone, with one CTA histogram each; the other CTAs read its answer. After a first
// pass over the whole cluster (first_pass = 1) the candidates are the members of the
// chosen top byte `prefix`: two cluster barriers instead of three histogram merges
// across the cluster, and the same tau, total above tau and count and mass of keys
// equal to tau as those merges would give. With first_pass = 0 the candidates are the
// whole set (top-k's survivors) and, when top_p >= 0, the mass target is formed here,
// ceil(top_p * their total mass) (at least 1), and returned in `target`.
__device__ uint32_t local_finish(const uint32_t *cand, int ncand, uint32_t *buf, uint32_t prefix,
                                 int first_pass, bool by_mass, double top_p,
                                 unsigned long long &target, unsigned long long &above,
                                 unsigned int &eq_cnt, unsigned long long &eq_mass,
                                 SmpShared &sh, int &slot) {
  const uint32_t C = gridDim.x, rank = cluster_rank();
  if (threadIdx.x == 0) sh.pub_n[slot] = (unsigned)ncand;
  cluster_sync_all();  // every CTA's candidates and count are published
  if (rank == 0) {
    // the cluster's candidates, CTA by CTA, into buf
    if (threadIdx.x == 0) {
      unsigned int n[kMaxCl];
#pragma unroll
      for (uint32_t q = 0; q < kMaxCl; ++q)
        if (q < C) n[q] = ld_cl_u32(map_rank(&sh.pub_n[slot], q));
      unsigned int off = 0;
#pragma unroll
      for (uint32_t q = 0; q < kMaxCl; ++q)
        if (q < C) {
          sh.warp_u64[q][0] = off;  // scratch: where CTA q's keys go
          sh.warp_u64[q][1] = n[q];
          off += n[q];
        }
      sh.bc_u32[2] = off;
    }
    __syncthreads();
    const int total = (int)sh.bc_u32[2];
    // every thread's loads (up to four keys, from any CTA) are issued before any is used
    constexpr int kPer = kCandCap / kSmpThreads;
    uint32_t key[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = threadIdx.x + j * kSmpThreads;
      if (i < total) {
        uint32_t q = 0;  // the CTA whose keys hold position i
        while (q + 1 < C && (int)sh.warp_u64[q + 1][0] <= i) ++q;
        const int k = i - (int)sh.warp_u64[q][0];
        key[j] = q == 0 ? cand[k] : ld_cl_u32(map_rank(&cand[k], q));
      }
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = threadIdx.x + j * kSmpThreads;
      if (i < total) buf[i] = key[j];
    }
    __syncthreads();
    if (top_p >= 0.0) {  // the target from the candidates' total mass
      unsigned long long m = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + j * kSmpThreads;
        if (i < total) m += to_mass(__uint_as_float(buf[i]));
      }
      unsigned long long mass;
      (void)block_exclusive_u64(m, sh, mass);
      target = (unsigned long long)ceil(top_p * (double)mass);
      if (target == 0) target = 1;
    }
    // one histogram for the CTA, past the candidates (at most kCandCap words) in the
    // same shared memory: at most 2^11 elements per pass keep its 32-bit sums exact
    WarpHist &hist = *reinterpret_cast<WarpHist *>(buf + kCandCap + 256);
    for (int pass = first_pass; pass < 4; ++pass) {
      const int fixed = 8 * pass, shift = 24 - fixed;
      for (int b = threadIdx.x; b < kBuckets; b += kSmpThreads) {
        hist.cnt[b] = 0;
        hist.lo[b] = 0;
        hist.hi[b] = 0;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kCandCap / kSmpThreads; ++j) {  // warp-uniform: hist_add is a warp op
        const int i = threadIdx.x + j * kSmpThreads;
        int b = kBuckets;
        unsigned long long m = 0;
        if (i < total) {
          const uint32_t key = buf[i];
          if (fixed == 0 || (key >> (32 - fixed)) == prefix) {
            b = (key >> shift) & 0xff;
            m = by_mass ? to_mass(__uint_as_float(key)) : 0ull;
          }
        }
        hist_add(hist, b, m);
      }
      __syncthreads();
      for (int b = threadIdx.x; b < kBuckets; b += kSmpThreads) {
        sh.cnt[b] = hist.cnt[b];
        sh.mass[b] = (unsigned long long)hist.lo[b] + ((unsigned long long)hist.hi[b] << 20);
      }
      __syncthreads();
      const int b = radix_pick(by_mass, target, above, eq_cnt, eq_mass, sh);
      prefix = (prefix << 8) | (uint32_t)b;
    }
    if (threadIdx.x == 0) {
      sh.pub_sel[slot][0] = prefix;
      sh.pub_sel[slot][1] = above;
      sh.pub_sel[slot][2] = ((unsigned long long)eq_cnt << 32) | 0u;
      sh.pub_u64[slot][0] = eq_mass;
      sh.pub_u64[slot][1] = target;
    }
  }
  cluster_sync_all();  // CTA 0's answer is published; it has read every candidate
  if (threadIdx.x == 0) {
    sh.bc_u64[0] = ld_cl_u64(map_rank(&sh.pub_sel[slot][0], 0));
    sh.bc_u64[1] = ld_cl_u64(map_rank(&sh.pub_sel[slot][1], 0));
    sh.bc_u64[2] = ld_cl_u64(map_rank(&sh.pub_sel[slot][2], 0));
    sh.bc_u64[3] = ld_cl_u64(map_rank(&sh.pub_u64[slot][0], 0));
    sh.warp_u64[0][1] = ld_cl_u64(map_rank(&sh.pub_u64[slot][1], 0));
  }
  __syncthreads();
  const uint32_t tau = (uint32_t)sh.bc_u64[0];
  above = sh.bc_u64[1];
  eq_cnt = (unsigned int)(sh.bc_u64[2] >> 32);
  eq_mass = sh.bc_u64[3];
  target = sh.warp_u64[0][1];
  __syncthreads();
  slot ^= 1;
  return tau;
}

// Full radix select (4 passes of 8 bits) over the members of `set`: the key tau of the
// element where the running total (count or mass) from the top first reaches `target`,
// the total strictly above tau, and the count and mass of the members equal to tau.
// With top_p >= 0 the mass target is formed from the first pass's cluster histogram,
// ceil(top_p * the members' total mass) (at least 1), and returned in `target`.
// The first pass walks the chunk in token-id order (membership depends on it). When the
// chosen top-byte bucket holds at most kCandCap members over the cluster, they are
// gathered into `cand` and local_finish ends the select on one CTA; otherwise three
// more passes walk the chunk again.
// `prebuilt`: the first pass's histograms were already filled (by the exponentials'
// loop, for a select over every token).
template <int G, typename Pred>
__device__ uint32_t radix_select(const float *vals, int c0, int c1, int per, Pred set,
                                 bool prebuilt, bool by_mass, double top_p,
                                 unsigned long long &target, unsigned long long &above,
                                 unsigned int &eq_cnt, unsigned long long &eq_mass,
                                 SmpShared &sh, WarpHist *wh, uint32_t *cand, int &slot) {
  const int lane = threadIdx.x & 31;
  WarpHist &mine = wh[(threadIdx.x >> 5) / (kSmpWarps / G)];
  above = 0;
  if (!prebuilt) {
    hist_clear<G>(wh);
    set.begin();
    for (int j = 0; j < per; ++j) {
      const int i = c0 + j;
      int b = kBuckets;
      unsigned long long m = 0;
      if (i < c1) {
        const float e = vals[padded(i)];
        const uint32_t key = __float_as_uint(e);
        if (set.next(key)) {
          b = key >> 24;
          m = by_mass ? to_mass(e) : 0ull;
        }
      }
      hist_add(mine, b, m);
    }
  }
  hist_merge<G>(wh, sh, slot);
  if (top_p >= 0.0) {  // the members' total mass is the histogram's
    if (threadIdx.x < 32) {
      unsigned long long t = 0;
#pragma unroll
      for (int j = 0; j < kBuckets / 32; ++j) t += sh.mass[threadIdx.x + 32 * j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (threadIdx.x == 0) {
        unsigned long long tg = (unsigned long long)ceil(top_p * (double)t);
        sh.bc_u64[3] = tg == 0 ? 1 : tg;
      }
    }
    __syncthreads();
    target = sh.bc_u64[3];
    __syncthreads();
  }
  uint32_t prefix = (uint32_t)radix_pick(by_mass, target, above, eq_cnt, eq_mass, sh);
  const bool gathered = eq_cnt <= (unsigned)kCandCap;  // the same on every CTA

  // gather the candidates of the chosen bucket
  if (threadIdx.x == 0) sh.bc_u32[1] = 0;
  __syncthreads();
  if (gathered) {
    set.begin();
    for (int j = 0; j < per; ++j) {
      const int i = c0 + j;
      bool take = false;
      uint32_t key = 0;
      if (i < c1) {
        key = __float_as_uint(vals[padded(i)]);
        take = set.next(key) && (key >> 24) == prefix;
      }
      const unsigned ball = __ballot_sync(0xffffffffu, take);
      unsigned base = 0;
      if (lane == 0 && ball) base = atomicAdd(&sh.bc_u32[1], (unsigned)__popc(ball));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (take) cand[base + __popc(ball & ((1u << lane) - 1u))] = key;
    }
    __syncthreads();
  }
  if (gathered)
    return local_finish(cand, (int)sh.bc_u32[1], reinterpret_cast<uint32_t *>(wh), prefix, 1,
                        by_mass, -1.0, target, above, eq_cnt, eq_mass, sh, slot);
  // not gathered (a flat row): the later passes walk the chunk again
  for (int pass = 1; pass < 4; ++pass) {
    const int fixed = 8 * pass, shift = 24 - fixed;
    hist_clear<G>(wh);
    set.begin();
    for (int j = 0; j < per; ++j) {
      int b = kBuckets;
      unsigned long long m = 0;
      const int i = c0 + j;
      if (i < c1) {
        const uint32_t key = __float_as_uint(vals[padded(i)]);
        if (set.next(key) && (key >> (32 - fixed)) == prefix) {
          b = (key >> shift) & 0xff;
          m = by_mass ? to_mass(__uint_as_float(key)) : 0ull;
        }
      }
      hist_add(mine, b, m);
    }
    hist_merge<G>(wh, sh, slot);
    const int b = radix_pick(by_mass, target, above, eq_cnt, eq_mass, sh);
    prefix = (prefix << 8) | (uint32_t)b;
  }
  __syncthreads();
  return prefix;
}

// The top-p select over top-k's survivors when there are at most kCandCap of them:
// every CTA gathers its members of `set` (walked in token-id order), CTA 0 forms the
// mass target from their total and runs all four 8-bit passes over them alone. The
// same answer as the cluster-wide select (every sum is an exact integer sum), without
// its pass over the whole row, its histogram merge and the cluster sum of the mass.
template <typename Pred>
__device__ uint32_t survivors_select(const float *vals, int c0, int c1, int per, Pred set,
                                     double top_p, unsigned long long &target,
                                     unsigned long long &above, unsigned int &eq_cnt,
                                     unsigned long long &eq_mass, SmpShared &sh, WarpHist *wh,
                                     uint32_t *cand, int &slot) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) sh.bc_u32[1] = 0;
  __syncthreads();
  set.begin();
  for (int j = 0; j < per; ++j) {  // warp-uniform trip count: the ballot is a warp op
    const int i = c0 + j;
    bool take = false;
    uint32_t key = 0;
    if (i < c1) {
      key = __float_as_uint(vals[padded(i)]);
      take = set.next(key);
    }
    const unsigned ball = __ballot_sync(0xffffffffu, take);
    unsigned base = 0;
    if (lane == 0 && ball) base = atomicAdd(&sh.bc_u32[1], (unsigned)__popc(ball));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (take) cand[base + __popc(ball & ((1u << lane) - 1u))] = key;
  }
  __syncthreads();
  above = 0;
  return local_finish(cand, (int)sh.bc_u32[1], reinterpret_cast<uint32_t *>(wh), 0u, 0, true,
                      top_p, target, above, eq_cnt, eq_mass, sh, slot);
}

template <int G>
__global__ void __launch_bounds__(kSmpThreads, G == kBatchGroups ? 2 : 1)
    sampler_kernel(const SmpArgs a) {
  extern __shared__ __align__(16) uint8_t smp_dyn[];
  // per-group histograms, the slice (padded), the radix-select candidates
  auto *wh = reinterpret_cast<WarpHist *>(smp_dyn);
  float *vals = reinterpret_cast<float *>(smp_dyn + G * sizeof(WarpHist));
  uint32_t *cand = reinterpret_cast<uint32_t *>(vals + a.slice + a.slice / 32);
  __shared__ SmpShared sh;
  __shared__ Member mem;
  const int row = blockIdx.y;
  const uint32_t rank = cluster_rank();
  const int lo = (int)rank * a.slice;
  const int n = max(0, min(a.V - lo, a.slice));
  const float *zrow = a.logits + (size_t)row * a.V;
  int slot = 0;

  pdl_launch_dependents();
  pdl_wait_prior_grid();

  // 1. load the slice, then the penalty from the original logits
  for (int i = threadIdx.x; i < n; i += kSmpThreads) vals[padded(i)] = zrow[lo + i];
  __syncthreads();
  if (a.ids != nullptr && a.penalty != 1.0f) {
    const int32_t *ids = a.ids + (size_t)row * a.L;
    for (int j = threadIdx.x; j < a.L; j += kSmpThreads) {
      const int id = ids[j];
      if (id >= lo && id < lo + n) {
        const float v = zrow[id];
        vals[padded(id - lo)] = v > 0.f ? v / a.penalty : v * a.penalty;
      }
    }
  }
  __syncthreads();

  const int per = (n + kSmpThreads - 1) / kSmpThreads;
  const int c0 = min(n, (int)threadIdx.x * per), c1 = min(n, c0 + per);

  // 2. greedy
  if (!(a.temperature > 0.f)) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = c0; i < c1; ++i) {
      const float v = vals[padded(i)];
      if (v > bv || i == c0) {  // the chunk is walked in id order: the first maximum wins
        bv = v;
        bi = lo + i;
      }
    }
    const int tok = cluster_argmax(bv, bi, sh, slot);
    if (rank == 0 && threadIdx.x == 0) a.tokens[row] = tok;
    cluster_sync_all();
    return;
  }

  // 2'. temperature, maximum, exponentials
  float mx = -INFINITY;
  for (int i = c0; i < c1; ++i) {
    const float z = vals[padded(i)] / a.temperature;
    vals[padded(i)] = z;
    mx = fmaxf(mx, z);
  }
  const float M = cluster_max(mx, sh, slot);
  const bool use_k = a.top_k > 0 && a.top_k < a.V, use_p = a.top_p < 1.0f;
  // The exponentials. When the first select covers every token (top-k by count, or
  // top-p by mass without a top-k), its first radix pass rides along.
  const bool first_all = use_k || use_p;
  const bool first_by_mass = !use_k;
  if (first_all) {
    WarpHist &mine = wh[(threadIdx.x >> 5) / (kSmpWarps / G)];
    hist_clear<G>(wh);
    for (int j = 0; j < per; ++j) {  // warp-uniform trip count: hist_add is a warp op
      const int i = c0 + j;
      int b = kBuckets;
      unsigned long long m = 0;
      if (i < c1) {
        const float e = expf(vals[padded(i)] - M);
        vals[padded(i)] = e;
        b = __float_as_uint(e) >> 24;
        m = first_by_mass ? to_mass(e) : 0ull;
      }
      hist_add(mine, b, m);
    }
  } else {
    for (int i = c0; i < c1; ++i) vals[padded(i)] = expf(vals[padded(i)] - M);
  }
  if (threadIdx.x == 0) {
    mem.use_k = use_k;
    mem.use_p = use_p;
    mem.tau_k = mem.tau_p = 0;
    mem.need_k = mem.need_p = 0;
  }
  __syncthreads();

  // 4. top-k: the k-th largest key, and how many of the keys equal to it are kept
  unsigned long long eqk_start = 0;
  if (mem.use_k) {
    struct All {
      __device__ void begin() {}
      __device__ bool next(uint32_t) { return true; }
    };
    unsigned long long above;
    unsigned int eq_cnt;
    unsigned long long eq_mass;
    unsigned long long kth = (unsigned long long)a.top_k;
    const uint32_t tau = radix_select<G>(vals, c0, c1, per, All{}, true, false, -1.0, kth,
                                      above, eq_cnt, eq_mass, sh, wh, cand, slot);
    const unsigned long long need = (unsigned long long)a.top_k - above;
    if (threadIdx.x == 0) {
      mem.tau_k = tau;
      mem.need_k = need;
    }
    __syncthreads();
    if (need < eq_cnt) {  // a tie straddles the cut: rank the equal keys by token id
      unsigned long long tot;
      const unsigned long long mine = count_equal(vals, c0, c1, tau, All{});
      const unsigned long long cta_before = block_exclusive_u64(mine, sh, tot);
      const unsigned long long cl_before = cluster_exclusive_u64(tot, sh, slot, tot);
      eqk_start = cl_before + cta_before;
    }
  }

  // 5. top-p over the top-k survivors
  unsigned long long eqp_start = 0;
  InK ink{&mem, eqk_start, 0};
  if (mem.use_p) {
    unsigned long long target = 0, above;
    unsigned int eq_cnt;
    unsigned long long eq_mass;
    uint32_t tau;
    if (use_k && a.top_k <= kCandCap) {  // few survivors: select among them on CTA 0
      tau = survivors_select(vals, c0, c1, per, ink, (double)a.top_p, target, above, eq_cnt,
                             eq_mass, sh, wh, cand, slot);
    } else {  // over the row's survivors; the target from the first pass's histogram
      tau = radix_select<G>(vals, c0, c1, per, ink, !use_k, true, (double)a.top_p, target,
                            above, eq_cnt, eq_mass, sh, wh, cand, slot);
    }
    const unsigned long long one = eq_cnt ? eq_mass / eq_cnt : 0;  // equal keys, equal mass
    unsigned long long need = eq_cnt;
    if (one > 0 && target > above) {
      need = (target - above + one - 1) / one;
      if (need < 1) need = 1;
      if (need > eq_cnt) need = eq_cnt;
    }
    if (threadIdx.x == 0) {
      mem.tau_p = tau;
      mem.need_p = need;
    }
    __syncthreads();
    if (need < eq_cnt) {  // a tie straddles the cut: rank the equal keys by token id
      unsigned long long tot2;
      const unsigned long long mine = count_equal(vals, c0, c1, tau, ink);
      const unsigned long long cta_before = block_exclusive_u64(mine, sh, tot2);
      const unsigned long long cl_before = cluster_exclusive_u64(tot2, sh, slot, tot2);
      eqp_start = cl_before + cta_before;
    }
  }

  // 6. the draw: first nucleus member, in token-id order, whose running mass > target
  InNucleus nuc{InK{&mem, eqk_start, 0}, &mem, eqp_start, 0};
  unsigned long long chunk = 0;
  nuc.begin();
  for (int i = c0; i < c1; ++i) {
    const float e = vals[padded(i)];
    if (nuc.next(__float_as_uint(e))) chunk += to_mass(e);
  }
  unsigned long long cta_tot;
  const unsigned long long t_before = block_exclusive_u64(chunk, sh, cta_tot);
  unsigned long long total;
  const unsigned long long c_before = cluster_exclusive_u64(cta_tot, sh, slot, total);
  const double uu = fmin(fmax((double)a.u[row], 0.0), 1.0);
  unsigned long long target = (unsigned long long)floor(uu * (double)total);
  if (total > 0 && target >= total) target = total - 1;
  const unsigned long long start = c_before + t_before;
  if (chunk > 0 && target >= start && target < start + chunk) {
    unsigned long long run = start;
    nuc.begin();
    for (int i = c0; i < c1; ++i) {
      const float e = vals[padded(i)];
      if (!nuc.next(__float_as_uint(e))) continue;
      run += to_mass(e);
      if (run > target) {
        a.tokens[row] = lo + i;
        break;
      }
    }
  }
  cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace

// CTAs per row: enough that a CTA holds at most 8192 logits, at most 16 (16 needs the
// non-portable cluster size, used when the device can place such clusters).
int sampler_cluster(int V) {
  int C = 1;
  while (C < 16 && (V + C - 1) / C > 8192) C *= 2;
  return C;
}

static int sampler_slice(int V, int C) {
  int slice = (V + C - 1) / C;
  return (slice + 31) & ~31;
}

static size_t smem_for(int V, int C, int G) {
  const int slice = sampler_slice(V, C);
  return (size_t)G * sizeof(WarpHist) + (size_t)(slice + slice / 32) * sizeof(float) +
         (size_t)kCandCap * sizeof(uint32_t);
}

static bool sampler_fits(int V, int C, int G) {
  return sampler_slice(V, C) <= max_slice(G) && smem_for(V, C, G) <= kSamplerMaxSmem;
}

bool sampler_supports(int V) {
  return V >= 1 && V <= 16 * max_slice(kBatchGroups) && sampler_fits(V, 16, kBatchGroups) &&
         sampler_fits(V, 16, kLatencyGroups);
}

// Clusters of C CTAs (shared memory smem each) of build G that the device holds at
// once, cached per device for the last few shapes.
template <int G>
static int resident_clusters(int dev, int C, size_t smem) {
  struct Entry {
    int dev, C;
    size_t smem;
    int n;
  };
  static Entry cache[16] = {};
  static std::atomic<int> next{0};
  for (const Entry &en : cache)
    if (en.n > 0 && en.dev == dev && en.C == C && en.smem == smem) return en.n;
  cudaLaunchConfig_t q = {};
  q.gridDim = dim3(C, 1, 1);
  q.blockDim = dim3(kSmpThreads);
  q.dynamicSmemBytes = smem;
  cudaLaunchAttribute qa[1];
  qa[0].id = cudaLaunchAttributeClusterDimension;
  qa[0].val.clusterDim.x = (unsigned)C;
  qa[0].val.clusterDim.y = 1;
  qa[0].val.clusterDim.z = 1;
  q.attrs = qa;
  q.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, sampler_kernel<G>, &q) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (n > 0) cache[next.fetch_add(1) & 15] = Entry{dev, C, smem, n};
  return n;
}

template <int G>
static cudaError_t sampler_attrs() {
  cudaError_t e = cudaFuncSetAttribute(sampler_kernel<G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSamplerMaxSmem);
  if (e != cudaSuccess) return e;
  // the largest shared-memory carveout, so that two batch CTAs fit on one SM
  e = cudaFuncSetAttribute(sampler_kernel<G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (cudaFuncSetAttribute(sampler_kernel<G>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) != cudaSuccess)
    (void)cudaGetLastError();  // clusters of up to 8 only
  return cudaSuccess;
}

cudaError_t launch_sampler(const float *logits, const int32_t *ids, int L, const float *u,
                           int32_t *tokens, int B, int V, float penalty, float temperature,
                           float top_p, int top_k, cudaStream_t stream) {
  static int attr_set[64] = {};  // 0 unknown, 1 set (clusters of 16 placeable), 2 set (not)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = (dev >= 0 && dev < 64) ? dev : 0;
  if (attr_set[di] == 0) {
    if ((e = sampler_attrs<kLatencyGroups>()) != cudaSuccess) return e;
    if ((e = sampler_attrs<kBatchGroups>()) != cudaSuccess) return e;
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(16, 1, 1);
    q.blockDim = dim3(kSmpThreads);
    q.dynamicSmemBytes = smem_for(1 << 17, 16, kLatencyGroups);
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = 16;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int n = 0;
    const bool placeable =
        cudaOccupancyMaxActiveClusters(&n, sampler_kernel<kLatencyGroups>, &q) == cudaSuccess &&
        n > 0;
    (void)cudaGetLastError();
    attr_set[di] = placeable ? 1 : 2;
  }
  const int cmax = attr_set[di] == 1 ? 16 : 8;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 1;
  // A few rows: sampler_cluster(V) CTAs per row (per-warp histograms) when every row's
  // cluster is resident at once, each CTA on an SM of its own. More rows: the batch
  // build, at the cluster size that keeps the most rows resident at once (as the
  // occupancy calculator places clusters), the larger size on a tie.
  int C = 0, G = kLatencyGroups;
  const int c_lat = sampler_cluster(V) < cmax ? sampler_cluster(V) : cmax;
  if ((long long)B * c_lat <= sms && sampler_fits(V, c_lat, kLatencyGroups) &&
      B <= resident_clusters<kLatencyGroups>(dev, c_lat, smem_for(V, c_lat, kLatencyGroups)))
    C = c_lat;
  if (C == 0) {
    G = kBatchGroups;
    int best_rows = 0;
    for (int c = cmax; c >= 1; c >>= 1) {
      if (!sampler_fits(V, c, kBatchGroups)) continue;
      const int rows = resident_clusters<kBatchGroups>(dev, c, smem_for(V, c, kBatchGroups));
      if (rows > best_rows) {
        best_rows = rows;
        C = c;
      }
    }
    if (C == 0) return cudaErrorInvalidValue;  // beyond this device's clusters
  }
  const int slice = sampler_slice(V, C);
  SmpArgs a{logits, ids, u, tokens, V, L, slice, penalty, temperature, top_p, top_k};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, B, 1);
  cfg.blockDim = dim3(kSmpThreads);
  cfg.dynamicSmemBytes = smem_for(V, C, G);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = G == kBatchGroups ? cudaLaunchKernelEx(&cfg, sampler_kernel<kBatchGroups>, a)
                        : cudaLaunchKernelEx(&cfg, sampler_kernel<kLatencyGroups>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace decattn
