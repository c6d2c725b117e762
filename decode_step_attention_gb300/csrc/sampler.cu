// The sampling side of a decode step, fused into one launch (fusedtok 1.0.1 README,
// "Operators": repetition penalty, temperature, argmax, sample_topk, sample_topp,
// decode_step = penalty -> temperature -> nucleus sample; "Usage": one call per step).
//
// One thread-block cluster of C CTAs per row of logits (C = 1, 2, 4 or 8): CTA r keeps
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
//      counts) finds the k-th largest value; equal values are ranked by token id;
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
#include <math.h>

#include "dec_device.cuh"
#include "dec_launch.h"

namespace decattn {
namespace {

constexpr int kSmpThreads = 512;
constexpr int kSmpWarps = kSmpThreads / 32;
constexpr int kBuckets = 256;

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
    unsigned long long before = 0, all = 0;
    for (uint32_t q = 0; q < C; ++q) {
      const unsigned long long v = ld_cl_u64(map_rank(&sh.pub_u64[slot][0], q));
      if (q < rank) before += v;
      all += v;
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
    float m = -INFINITY;
    for (uint32_t q = 0; q < gridDim.x; ++q) m = fmaxf(m, ld_cl_f32(map_rank(&sh.pub_f[slot], q)));
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
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (uint32_t q = 0; q < gridDim.x; ++q) {
      const float qv = ld_cl_f32(map_rank(&sh.pub_f[slot], q));
      const int qi = (int)ld_cl_u32(map_rank(&sh.pub_i[slot], q));
      if (qv > bv || (qv == bv && qi < bi)) {
        bv = qv;
        bi = qi;
      }
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

// One radix-select pass over this CTA's chunk: histogram (count and mass) of the keys
// of the candidates whose top `fixed` bits equal `prefix`, bucketed by the next 8 bits;
// then the cluster's histogram (the sum over CTAs, in rank order) in sh.cnt / sh.mass.
// The lanes of a warp walk their chunks in step; lanes that hit the same bucket are
// combined first (__match_any_sync, then __reduce_add_sync of the count and of the
// mass split into two 21-bit halves, so the integer sums stay exact), and each warp
// adds into its own histogram, so no two warps contend for a bucket.
template <typename Pred>
__device__ void radix_histogram(const float *vals, int c0, int c1, int per, uint32_t prefix,
                                int fixed, Pred in_set, SmpShared &sh,
                                unsigned int (*wcnt)[kBuckets],
                                unsigned long long (*wmass)[kBuckets], int &slot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = lane; b < kBuckets; b += 32) {
    wcnt[warp][b] = 0;
    wmass[warp][b] = 0;
  }
  __syncwarp();
  const int shift = 24 - fixed;
  in_set.begin();
  for (int j = 0; j < per; ++j) {
    const int i = c0 + j;
    int b = kBuckets;  // not counted
    unsigned long long m = 0;
    if (i < c1) {
      const float e = vals[padded(i)];
      const uint32_t key = __float_as_uint(e);
      if (in_set.next(key) && (fixed == 0 || (key >> (32 - fixed)) == prefix)) {
        b = (key >> shift) & 0xff;
        m = to_mass(e);
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    if (b < kBuckets) {
      const unsigned lo = __reduce_add_sync(peers, (unsigned)(m & 0x1FFFFFull));
      const unsigned hi = __reduce_add_sync(peers, (unsigned)(m >> 21));
      if (lane == __ffs(peers) - 1) {
        wcnt[warp][b] += __popc(peers);
        wmass[warp][b] += (unsigned long long)lo + ((unsigned long long)hi << 21);
      }
    }
    __syncwarp();
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kBuckets; b += kSmpThreads) {
    unsigned int c = 0;
    unsigned long long ms = 0;
    for (int w = 0; w < kSmpWarps; ++w) {
      c += wcnt[w][b];
      ms += wmass[w][b];
    }
    sh.pub_cnt[slot][b] = c;
    sh.pub_mass[slot][b] = ms;
  }
  cluster_sync_all();
  for (int b = threadIdx.x; b < kBuckets; b += kSmpThreads) {
    unsigned int c = 0;
    unsigned long long ms = 0;
    for (uint32_t q = 0; q < gridDim.x; ++q) {
      c += ld_cl_u32(map_rank(&sh.pub_cnt[slot][b], q));
      ms += ld_cl_u64(map_rank(&sh.pub_mass[slot][b], q));
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

// Full radix select (4 passes) over the members of `set`: the key tau of the element
// where the running total (count or mass) from the top first reaches `target`, the
// total strictly above tau, and the count and mass of the members equal to tau.
template <typename Pred>
__device__ uint32_t radix_select(const float *vals, int c0, int c1, int per, Pred set,
                                 bool by_mass, unsigned long long target,
                                 unsigned long long &above, unsigned int &eq_cnt,
                                 unsigned long long &eq_mass, SmpShared &sh,
                                 unsigned int (*wcnt)[kBuckets],
                                 unsigned long long (*wmass)[kBuckets], int &slot) {
  uint32_t prefix = 0;
  above = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int fixed = 8 * pass;
    radix_histogram(vals, c0, c1, per, prefix, fixed, set, sh, wcnt, wmass, slot);
    const int b = radix_pick(by_mass, target, above, eq_cnt, eq_mass, sh);
    prefix = (prefix << 8) | (uint32_t)b;
  }
  return prefix;
}

__global__ void __launch_bounds__(kSmpThreads) sampler_kernel(const SmpArgs a) {
  extern __shared__ __align__(16) uint8_t smp_dyn[];
  // per-warp histograms, then the slice (padded)
  auto *wmass = reinterpret_cast<unsigned long long (*)[kBuckets]>(smp_dyn);
  auto *wcnt = reinterpret_cast<unsigned int (*)[kBuckets]>(smp_dyn + kSmpWarps * kBuckets * 8);
  float *vals = reinterpret_cast<float *>(smp_dyn + kSmpWarps * kBuckets * 12);
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
  for (int i = c0; i < c1; ++i) vals[padded(i)] = expf(vals[padded(i)] - M);
  __syncthreads();

  if (threadIdx.x == 0) {
    mem.use_k = a.top_k > 0 && a.top_k < a.V;
    mem.use_p = a.top_p < 1.0f;
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
    const uint32_t tau = radix_select(vals, c0, c1, per, All{}, false,
                                      (unsigned long long)a.top_k, above, eq_cnt, eq_mass, sh,
                                      wcnt, wmass, slot);
    if (threadIdx.x == 0) {
      mem.tau_k = tau;
      mem.need_k = (unsigned long long)a.top_k - above;
    }
    __syncthreads();
    // equal keys before this chunk, in token-id order
    unsigned long long tot;
    const unsigned long long mine = count_equal(vals, c0, c1, tau, All{});
    const unsigned long long cta_before = block_exclusive_u64(mine, sh, tot);
    const unsigned long long cl_before = cluster_exclusive_u64(tot, sh, slot, tot);
    eqk_start = cl_before + cta_before;
  }

  // 5. top-p over the top-k survivors
  unsigned long long eqp_start = 0;
  InK ink{&mem, eqk_start, 0};
  if (mem.use_p) {
    // the survivors' mass
    unsigned long long mk = 0;
    ink.begin();
    for (int i = c0; i < c1; ++i) {
      const float e = vals[padded(i)];
      if (ink.next(__float_as_uint(e))) mk += to_mass(e);
    }
    unsigned long long tot;
    (void)block_exclusive_u64(mk, sh, tot);
    unsigned long long mass_k;
    (void)cluster_exclusive_u64(tot, sh, slot, mass_k);
    const double tp = (double)a.top_p * (double)mass_k;
    unsigned long long target = (unsigned long long)ceil(tp);
    if (target == 0) target = 1;
    unsigned long long above;
    unsigned int eq_cnt;
    unsigned long long eq_mass;
    const uint32_t tau = radix_select(vals, c0, c1, per, ink, true, target, above, eq_cnt,
                                      eq_mass, sh, wcnt, wmass, slot);
    if (threadIdx.x == 0) {
      mem.tau_p = tau;
      const unsigned long long one = eq_cnt ? eq_mass / eq_cnt : 0;  // equal keys, equal mass
      unsigned long long need = eq_cnt;
      if (one > 0 && target > above) {
        need = (target - above + one - 1) / one;
        if (need < 1) need = 1;
        if (need > eq_cnt) need = eq_cnt;
      }
      mem.need_p = need;
    }
    __syncthreads();
    unsigned long long tot2;
    const unsigned long long mine = count_equal(vals, c0, c1, tau, ink);
    const unsigned long long cta_before = block_exclusive_u64(mine, sh, tot2);
    const unsigned long long cl_before = cluster_exclusive_u64(tot2, sh, slot, tot2);
    eqp_start = cl_before + cta_before;
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

int sampler_cluster(int V) {
  return V <= 4096 ? 1 : V <= 16384 ? 2 : V <= 65536 ? 4 : 8;
}

size_t sampler_smem(int V) {
  const int C = sampler_cluster(V);
  int slice = (V + C - 1) / C;
  slice = (slice + 31) & ~31;
  return (size_t)kSmpWarps * kBuckets * 12 + (size_t)(slice + slice / 32) * sizeof(float);
}

cudaError_t launch_sampler(const float *logits, const int32_t *ids, int L, const float *u,
                           int32_t *tokens, int B, int V, float penalty, float temperature,
                           float top_p, int top_k, cudaStream_t stream) {
  const int C = sampler_cluster(V);
  int slice = (V + C - 1) / C;
  slice = (slice + 31) & ~31;
  const size_t smem = sampler_smem(V);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(sampler_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSamplerMaxSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  SmpArgs a{logits, ids, u, tokens, V, L, slice, penalty, temperature, top_p, top_k};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, B, 1);
  cfg.blockDim = dim3(kSmpThreads);
  cfg.dynamicSmemBytes = smem;
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
  e = cudaLaunchKernelEx(&cfg, sampler_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace decattn
