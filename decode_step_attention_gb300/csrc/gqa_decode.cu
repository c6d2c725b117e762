// K3 + K4: single-query GQA decode attention over a contiguous bf16 KV cache.
//
// fusedtok README, "Operators" (attention_decode: single-token causal attention
// with GQA over a contiguous kv-cache, online softmax, flash-decoding split over
// long caches, per-sequence lengths) and "Usage" (q [B,Hq,D], caches [B,Hkv,T,D],
// lens [B] int32); "Benchmarks" (one launch streams the GQA cache once; heads are
// expanded with repeat_interleave, so query head h reads KV head h / G).
//
// Split pass (K3). The Hkv * sum(lens) rows (sequence b, KV head g, token t) are read
// as one stream, ordered by (b, g, t), and cut into pieces (PieceSched): one large
// piece per CTA, and small pieces that CTAs claim from a counter as they finish, so
// the SMs that get more bandwidth do more of the work and all finish together. A
// piece that crosses a (b, g) boundary yields one partial per pair it touches,
// stored in slot piece + b*Hkv + g (distinct for every touching (piece, pair),
// since pieces and pairs are both contiguous runs of the stream).
//
// Inside a CTA one producer lane walks its pieces and, per 128-token tile, writes a
// small descriptor and issues 128B-swizzled bulk-tensor (TMA) loads of the K and V
// tile (plus the group's queries on the first tile of a pair) into a ring of
// shared-memory stages guarded by mbarriers; the last partial tile of a run is
// loaded in 8-row boxes past its last whole 64-row box, so little is read past its
// end. Eight consumer warps each own 16 rows of a tile and serve all G <= 8 query
// heads of the KV head from that one read:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T        (mma m16n8k16, bf16 -> fp32)
//   online softmax per head column (base-2 exponent, running max and sum)
//   O^T[D x 8 heads]     += V^T[D x 16] . P^T      (P split into bf16 hi + lo parts,
//                                                   two mma, ~16-bit weights)
// The S^T accumulator layout turns into the P^T operand layout with one 8x8
// register transpose (movmatrix), so P never touches shared memory. At the end of a
// run the warps' (m, l, O) are combined through shared memory and the partial
// (normalised o and lse, base 2) is written.
//
// With a sliding window of W tokens (cutileGPT README, "The current runtime includes":
// sliding-window attention) a sequence contributes its last min(len, W) rows: the
// stream and every offset use that length and the loads start at row len - W.
//
// Merge (K4). For each query head, the partials of its (b, g) pair (pieces
// piece_of(first row) .. piece_of(last row)) are combined with log-sum-exp weights
// by a group of warps. With at most one CTA per SM the merge runs inside the split
// pass's own (cooperative) launch: each CTA marks its pieces done with the launch's
// epoch once it has streamed them, then merges heads as their pieces are marked
// (merge_phase). Otherwise it is a launch of its own (split_merge_kernel), reading the
// sequence offsets from the workspace, where the split pass left them.
#include <math.h>

#include "dec_device.cuh"
#include "dec_launch.h"

namespace decattn {
namespace {

constexpr int kTile = kSplitTile;        // tokens per stage
constexpr int kSubRows = 8;              // rows per box of a partial tile
constexpr int kConsumerWarps = 8;        // 8 warps x 16 rows = one tile
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kMaxStages = 8;
constexpr int kPrefetchTiles = 4;  // tiles a CTA prefetches into L2 before its wait

constexpr uint32_t kFirst = 1u, kLast = 2u, kEnd = 4u, kPieceEnd = 8u;
constexpr int kPieceList = 32;

// What the producer tells the consumers about the tile in a stage. 16-byte aligned
// size, so that the mbarriers placed after the stages' records stay 8-byte aligned.
struct alignas(16) TileMeta {
  int b, g;
  int tok0;     // first token of the tile within the pair
  int tok_end;  // end (exclusive) of the run the tile belongs to
  int L;        // length of sequence b
  int nload;    // rows actually loaded into the stage
  int slot;     // partial slot of the run
  int piece;    // the piece the tile belongs to
  uint32_t flags;
};

// Workspace header words (bytes 0..255): the device error word, the claim counter of
// the small pieces and the count of CTAs done claiming (both back at zero after every
// completed split pass), the direct-output flag, and for the one-launch attention the
// count of CTAs that have finished and the claim counter of the merge's work (both
// back at zero after every launch) and the launch epoch (one more after every launch;
// pieces of this launch are marked with it).
constexpr int kHdrError = 0, kHdrNextPiece = 1, kHdrDone = 2, kHdrDirect = 3;
constexpr int kHdrDepart = 5, kHdrMergeNext = 6, kHdrEpoch = 7;

template <int D>
struct Geom {
  static constexpr int kBoxes = D / 64;           // 128-byte swizzle boxes per row
  static constexpr int kBoxBytes = kTile * 128;   // one box of one tile
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
  static constexpr int kOStride = D + 4;          // floats between heads in the combine area
};

// Shared-memory layout of the split kernel (offsets from a 1024-aligned base).
struct SplitLayout {
  int stages, q_stride, q_off, meta_off, bar_off, scratch_off, warp_scratch, prefix_off, bytes;
};

__host__ __device__ inline SplitLayout split_layout(int D, int G, int B, int stages) {
  SplitLayout s;
  s.stages = stages;
  const int stage_bytes = 2 * (D / 64) * kTile * 128;
  s.q_stride = (G * D * 2 + 127) & ~127;
  s.q_off = stages * stage_bytes;
  s.meta_off = s.q_off + stages * s.q_stride;
  s.bar_off = s.meta_off + stages * (int)sizeof(TileMeta);  // a multiple of 16
  static_assert(sizeof(TileMeta) % 16 == 0, "mbarriers after the records need alignment");
  // full, empty, the consumers' rendezvous, the scratch's release; 16-byte reads of it
  s.scratch_off = (s.bar_off + (2 * stages + 2) * 8 + 15) & ~15;
  s.warp_scratch = (G * (D + 4) + 2 * G + 3) & ~3;  // floats, a multiple of four
  // the warps' states (each warp: o [G][D + 4], then m [G], then l [G])
  s.prefix_off = s.scratch_off + kConsumerWarps * s.warp_scratch * 4;
  s.bytes = 1024 + s.prefix_off + (B + 1) * 4 + 16;
  return s;
}

// A run of one (b, g) pair's tokens [t0, t1) inside a piece.
struct Seg {
  int b, g, t0, t1;
  long long r;   // stream row of t0
};

__device__ __forceinline__ int seq_len(const int *prefix, int b) { return prefix[b + 1] - prefix[b]; }

// First run of the piece [r0, r1) (r0 < r1 <= total).
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

// Shared address of (row, 16-byte chunk) of a tile written by SWIZZLE_128B TMA boxes:
// chunk c of row r lands at chunk c ^ (r & 7) of that row's 128 bytes.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * Geom<D>::kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait, bounded in time, until every non-empty piece of [c0, c1] (c1 < c0: none) is
// marked done in this launch. Called by a whole warp: each lane checks every 32nd
// piece, so the marks are read in parallel; they are read with acquire semantics, so
// the pieces' partials are visible afterwards. false: the wait gave up.
__device__ bool wait_pieces(const uint32_t *done, const PieceSched &sched, unsigned c0,
                            unsigned c1, uint32_t mark) {
  const unsigned lane = threadIdx.x & 31u;
  unsigned long long t0 = 0;
  while (true) {
    bool mine = true;
    if (c1 + 1 > c0)
      for (unsigned c = c0 + lane; c <= c1; c += 32)
        if (!sched.empty32(c) && ld_acquire_gpu(done + c) != mark) mine = false;
    if (__all_sync(0xffffffffu, mine)) {
      __syncwarp();  // every lane's later loads follow every lane's acquire
      return true;
    }
    if (t0 == 0) t0 = global_ns();
    else if (global_ns() - t0 > kWaitLimitNs) return false;
    __nanosleep(128);
  }
}

// The same for the pieces c, c + stride, ... (count of them, those past c1 or empty
// skipped): lane x checks piece c + x * stride.
__device__ bool wait_strided(const uint32_t *done, const PieceSched &sched, unsigned c,
                             unsigned stride, int count, unsigned c1, uint32_t mark) {
  const unsigned lane = threadIdx.x & 31u;
  const unsigned cc = c + lane * stride;
  const bool needed = lane < (unsigned)count && cc <= c1 && !sched.empty32(cc);
  unsigned long long t0 = 0;
  while (true) {
    const bool mine = !needed || ld_acquire_gpu(done + cc) == mark;
    if (__all_sync(0xffffffffu, mine)) {
      __syncwarp();
      return true;
    }
    if (t0 == 0) t0 = global_ns();
    else if (global_ns() - t0 > kWaitLimitNs) return false;
    __nanosleep(64);
  }
}

// The end of a launch: the last CTA to finish resets the count and moves the epoch on
// for the next launch (which cannot start before this one has finished).
__device__ void launch_depart(uint32_t *hdr, uint32_t nctas) {
  if (atomicAdd(hdr + kHdrDepart, 1u) == nctas - 1) {
    atomicExch(hdr + kHdrDepart, 0u);
    atomicExch(hdr + kHdrMergeNext, 0u);
    atomicAdd(hdr + kHdrEpoch, 1u);
  }
}

// Running log-sum-exp state of one query head's merge, per lane (E of the head's D
// values): the largest lse seen, the sum of 2^(lse - m), and the weighted o.
template <int E>
struct MergeAcc {
  float m, w, a[E];
  __device__ void init() {
    m = -INFINITY;
    w = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) a[e] = 0.f;
  }
  // fold in a partial (lse l, this lane's slice v of its o); l = -inf adds nothing
  __device__ void add(float l, const float (&v)[E]) {
    if (l == -INFINITY) return;
    const float mn = fmaxf(m, l);
    const float sc = exp2f(m - mn), f = exp2f(l - mn);
    w = w * sc + f;
#pragma unroll
    for (int e = 0; e < E; ++e) a[e] = a[e] * sc + f * v[e];
    m = mn;
  }
};

template <int E>
__device__ __forceinline__ void load_o(const float *p, float (&v)[E]) {
  if constexpr (E == 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4 *>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const float2 x = __ldcg(reinterpret_cast<const float2 *>(p));
    v[0] = x.x; v[1] = x.y;
  }
}

template <int E>
__device__ __forceinline__ void store_head(__nv_bfloat16 *orow, const MergeAcc<E> &acc) {
  const float inv = acc.w > 0.f ? 1.f / acc.w : 0.f;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(orow) = make_uint2(pack_bf16x2(acc.a[0] * inv, acc.a[1] * inv),
                                                  pack_bf16x2(acc.a[2] * inv, acc.a[3] * inv));
  } else {
    *reinterpret_cast<uint32_t *>(orow) = pack_bf16x2(acc.a[0] * inv, acc.a[1] * inv);
  }
}

// The merge of every query head whose pair spans several pieces, run by every thread
// of every CTA after the grid barrier of the one-launch attention. Partials are read
// through L2 (where the other CTAs wrote them) and folded into a running log-sum-exp
// state, so every load of a group of partials is in flight at once: one round of L2
// latency per group instead of two per partial. Pairs of a few pieces (wph = 1): each
// consumer warp merges kBatch heads at a time. Longer pairs: a CTA's wph warps share
// one head (wph = 8: the whole CTA) and combine through `scratch`.
template <int D>
__device__ __forceinline__ bool merge_heads(uint32_t *hdr, const uint8_t *workspace,
                                            const int *prefix, const PieceSched &sched,
                                            float *scratch, __nv_bfloat16 *out, int B, int Hq,
                                            int Hkv, int G, int wph, uint32_t mark) {
  constexpr int E = D / 32;  // floats per lane
  constexpr int kChunk = 8;  // partials of one head with loads in flight together
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = gridDim.x;
  const float *o_ws = reinterpret_cast<const float *>(workspace + kWsHeaderBytes);
  const float *lse_ws =
      reinterpret_cast<const float *>(workspace + ws_lse_offset(P, B, Hkv, G, D));
  const unsigned nheads = (unsigned)B * (unsigned)Hq;
  const uint32_t *done = reinterpret_cast<const uint32_t *>(
      workspace + ws_flags_offset(P, B, Hkv, G, D));
  bool ok = true;
  // the pieces [c0, c1] of a head's pair; c1 < c0 when the split pass wrote the head
  // itself (a pair in one piece); an empty sequence is written as zeros
  auto range = [&](unsigned head, unsigned &c0, unsigned &c1, size_t &pair, int &hh) -> bool {
    const int b = (int)(head / (unsigned)Hq), h = (int)(head - (unsigned)b * Hq);
    const int pre = prefix[b], Lb = prefix[b + 1] - pre;
    const int g = h / G;
    hh = h - g * G;
    pair = (size_t)b * Hkv + g;
    c0 = 1;
    c1 = 0;
    if (Lb > 0) {
      const unsigned st = (unsigned)Hkv * (unsigned)pre + (unsigned)g * (unsigned)Lb;
      c0 = sched.piece_of32(st);
      c1 = sched.piece_of32(st + Lb - 1);
      if (c1 == c0) return false;
    }
    return true;
  };
  auto slot_of = [&](unsigned c, size_t pair) { return (size_t)c + pair; };

  if (wph == 1) {
    // every warp of the CTA, the producer's included, claims kBatch consecutive heads
    // at a time from a counter: the CTAs that finish streaming first take most of the
    // work, and the last one to finish finds little left
    constexpr int kBatch = 2;
    while (true) {
      unsigned base = 0;
      if (lane == 0) base = atomicAdd(hdr + kHdrMergeNext, 1u) * kBatch;
      base = __shfl_sync(0xffffffffu, base, 0);
      if (base >= nheads) break;
      unsigned c0[kBatch], c1[kBatch];
      size_t pair[kBatch];
      int hh[kBatch];
      bool write[kBatch];
      MergeAcc<E> acc[kBatch];
      unsigned most = 0;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const unsigned head = base + k;
        acc[k].init();
        write[k] = head < nheads && range(head, c0[k], c1[k], pair[k], hh[k]);
        if (!write[k]) { c0[k] = 1; c1[k] = 0; pair[k] = 0; hh[k] = 0; }
        if (c1[k] + 1 > c0[k]) most = max(most, c1[k] + 1 - c0[k]);
      }
      // merge as soon as the heads' pieces are done (most are, long before the last CTA
      // finishes streaming)
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (ok && !wait_pieces(done, sched, c0[k], c1[k], mark)) ok = false;
      if (!ok) return false;
      for (unsigned j = 0; j < most; j += kChunk) {
        float l[kBatch][kChunk], v[kBatch][kChunk][E];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
#pragma unroll
          for (int x = 0; x < kChunk; ++x) {  // every load of the group first
            const unsigned c = c0[k] + j + x;
            l[k][x] = -INFINITY;
#pragma unroll
            for (int e = 0; e < E; ++e) v[k][x][e] = 0.f;
            if (c <= c1[k] && c1[k] + 1 > c0[k] && !sched.empty32(c)) {
              const size_t slot = slot_of(c, pair[k]);
              l[k][x] = __ldcg(lse_ws + slot * G + hh[k]);
              load_o<E>(o_ws + (slot * G + hh[k]) * D + lane * E, v[k][x]);
            }
          }
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
#pragma unroll
          for (int x = 0; x < kChunk; ++x) acc[k].add(l[k][x], v[k][x]);
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (write[k]) store_head<E>(out + (size_t)(base + k) * D + lane * E, acc[k]);
    }
    return ok;
  }

  // long pairs: wph warps per head, kConsumerWarps / wph heads per CTA at a time
  float *s_acc = scratch;                       // [8][D]
  float *s_m = scratch + kConsumerWarps * D;    // [8]
  float *s_w = s_m + kConsumerWarps;            // [8]
  const int hpc = kConsumerWarps / wph;
  const unsigned units = (nheads + hpc - 1) / hpc;
  const int hs = warp / wph, sub = warp - hs * wph;
  __shared__ unsigned s_unit;
  while (true) {
    if (threadIdx.x == 0) s_unit = atomicAdd(hdr + kHdrMergeNext, 1u);
    __syncthreads();
    const unsigned u = s_unit;
    if (u >= units) break;
    const unsigned head = u * hpc + hs;
    bool work = false;
    MergeAcc<E> acc;
    acc.init();
    if (warp < kConsumerWarps && head < nheads) {
      unsigned c0, c1;
      size_t pair;
      int hh;
      work = range(head, c0, c1, pair, hh);
      if (work && c1 >= c0) {
        // each chunk as soon as its own pieces are done: what is left when the last
        // piece of the pair is marked is the one chunk that holds it
        for (unsigned c = c0 + sub; c <= c1 && ok; c += kChunk * wph) {
          if (!wait_strided(done, sched, c, (unsigned)wph, kChunk, c1, mark)) {
            ok = false;
            break;
          }
          float l[kChunk], v[kChunk][E];
#pragma unroll
          for (int x = 0; x < kChunk; ++x) {
            const unsigned cc = c + x * wph;
            l[x] = -INFINITY;
#pragma unroll
            for (int e = 0; e < E; ++e) v[x][e] = 0.f;
            if (cc <= c1 && !sched.empty32(cc)) {
              const size_t slot = slot_of(cc, pair);
              l[x] = __ldcg(lse_ws + slot * G + hh);
              load_o<E>(o_ws + (slot * G + hh) * D + lane * E, v[x]);
            }
          }
#pragma unroll
          for (int x = 0; x < kChunk; ++x) acc.add(l[x], v[x]);
        }
      }
      if (lane == 0) { s_m[warp] = acc.m; s_w[warp] = acc.w; }
#pragma unroll
      for (int e = 0; e < E; ++e) s_acc[warp * D + lane * E + e] = acc.a[e];
    }
    __syncthreads();
    if (work && sub == 0) {
      MergeAcc<E> tot;
      tot.init();
      for (int w = 0; w < wph; ++w) {
        const int ww = hs * wph + w;
        const float mw = s_m[ww];
        if (mw == -INFINITY) continue;
        // fold warp ww's state (m, w, a) in as a partial of weight w at lse m
        const float mn = fmaxf(tot.m, mw);
        const float sc = exp2f(tot.m - mn), f = exp2f(mw - mn);
        tot.w = tot.w * sc + f * s_w[ww];
#pragma unroll
        for (int e = 0; e < E; ++e) tot.a[e] = tot.a[e] * sc + f * s_acc[ww * D + lane * E + e];
        tot.m = mn;
      }
      store_head<E>(out + (size_t)head * D + lane * E, tot);
    }
    __syncthreads();
  }
  return ok;
}

// The end of the one-launch attention, run by every thread of every CTA once it has
// streamed its pieces: the merge of every head whose pair spans several pieces, each as
// soon as the pieces it needs are marked done, then the departure that readies the
// workspace for the next launch.
template <int D>
__device__ __noinline__ void merge_phase(uint32_t *hdr, const uint8_t *workspace,
                                         const int *prefix, const PieceSched &sched,
                                         float *scratch, __nv_bfloat16 *out, int B, int Hq,
                                         int Hkv, int G, int wph, uint32_t mark,
                                         const int *pieces, int npieces) {
  __syncthreads();
  if (threadIdx.x == 0) {  // every consumer's partials of these pieces, then the marks
    fence_acq_rel_gpu();
    uint32_t *done = reinterpret_cast<uint32_t *>(
        const_cast<uint8_t *>(workspace) + ws_flags_offset(gridDim.x, B, Hkv, G, D));
    for (int i = 0; i < npieces; ++i) st_relaxed_gpu(done + pieces[i], mark);
  }
  if (!merge_heads<D>(hdr, workspace, prefix, sched, scratch, out, B, Hq, Hkv, G, wph, mark))
    atomicOr(hdr + kHdrError, kErrWaitTimeout);
  __syncthreads();
  if (threadIdx.x == 0) launch_depart(hdr, gridDim.x);
}

// kFused: the split pass and its merge in one launch. A CTA marks each piece done
// once its runs' partials are written; once it has streamed its own pieces, it merges
// its share of the query heads whose pairs span several pieces (merge_wph warps per
// head), each as soon as that pair's pieces are marked, reading the partials from L2;
// heads of pairs that lie in one piece were written by the split pass itself.
//
// kMode: 0 the split pass alone, 1 the split pass and its merge (kFused).
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1) gqa_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap kmap8, const __grid_constant__ CUtensorMap vmap8,
    const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ lens, int B, int Hq,
    int Hkv, int T_cap, float scale_log2, int stages, uint8_t *__restrict__ workspace,
    __nv_bfloat16 *__restrict__ out_direct, int window, int merge_wph) {
  constexpr bool kFused = kMode >= 1;
  constexpr int kNT = kThreads;
  using Gm = Geom<D>;
  constexpr int KS = D / 16;  // k-steps of S^T = K Q^T
  constexpr int MT = D / 16;  // m-tiles of O^T = V^T P^T
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_warp_tot[kNT / 32];
  __shared__ volatile int s_abort;
  // the pieces this CTA streams (its large piece and the small ones it claims), marked
  // done together once it has finished them; pieces past the list's end are marked
  // one by one as their last run closes
  __shared__ int s_pieces[kPieceList];
  __shared__ int s_npieces;

  const int G = Hq / Hkv;
  const SplitLayout lay = split_layout(D, G, B, stages);
  // 1024-byte aligned in the shared window; indexing off the __shared__ array keeps the
  // compiler's knowledge that this is shared memory (shared loads and stores rather than
  // generic ones)
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar_full = s_base + lay.bar_off;            // stages x 8 bytes
  const uint32_t bar_empty = bar_full + stages * 8;          // stages x 8 bytes
  const uint32_t bar_fin = bar_empty + stages * 8;           // consumer rendezvous
  const uint32_t bar_free = bar_fin + 8;  // every consumer warp is done reading the scratch
  TileMeta *meta = reinterpret_cast<TileMeta *>(smem + lay.meta_off);
  float *scratch = reinterpret_cast<float *>(smem + lay.scratch_off);
  int *prefix = reinterpret_cast<int *>(smem + lay.prefix_off);
  uint32_t *hdr = reinterpret_cast<uint32_t *>(workspace);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    mbar_init(bar_fin, kConsumerWarps);
    mbar_init(bar_free, kConsumerWarps);
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&kmap8);
    tma_prefetch_desc(&vmap8);
  }
  pdl_launch_dependents();
  // Until the wait for the previous kernel below, only inputs no kernel of the step
  // writes are read (the lengths, the cache rows through L2 prefetches), and nothing is
  // written outside shared memory: this part overlaps the previous kernel's tail.

  // ---- prologue: clamped lengths -> exclusive prefix sums in shared memory
  bool clamped = false;
  {
    const int chunk = (B + kNT - 1) / kNT;
    const int b0 = min(B, tid * chunk), b1 = min(B, b0 + chunk);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      int L = lens[b];
      if (L < 0 || L > T_cap) { clamped = true; L = L < 0 ? 0 : T_cap; }
      if (window > 0 && L > window) L = window;  // a sliding window keeps the last rows
      local += L;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp_tot[warp] = incl;
    if (tid == 0) { s_abort = 0; s_npieces = 0; }
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp_tot[w];
    int run = before + incl - local;
    for (int b = b0; b < b1; ++b) {
      prefix[b] = run;
      int L = lens[b];
      L = L < 0 ? 0 : (L > T_cap ? T_cap : L);
      if (window > 0 && L > window) L = window;
      run += L;
    }
    if (tid == kNT - 1) prefix[B] = before + incl;
  }
  __syncthreads();

  const long long total = (long long)Hkv * prefix[B];
  const PieceSched sched = PieceSched::make(total, gridDim.x);
  if (warp == kConsumerWarps && lane == 0) {
    // the first tiles of this CTA's large piece into L2 while the previous kernel ends
    // (L2 keeps them coherent with any slot that kernel still writes)
    const long long r0 = sched.start((long long)blockIdx.x * kPiecesPerBlock);
    const long long r1 = sched.start((long long)blockIdx.x * kPiecesPerBlock + 1);
    if (r0 < r1) {
      Seg sg = first_seg(prefix, B, Hkv, r0, r1);
      int left = kPrefetchTiles;
      do {
        int Lfull = lens[sg.b];
        Lfull = Lfull < 0 ? 0 : (Lfull > T_cap ? T_cap : Lfull);
        const int base = Lfull - seq_len(prefix, sg.b);
        const int pair = sg.b * Hkv + sg.g;
        for (int tt = sg.t0; tt < sg.t1 && left > 0; tt += kTile, --left)
          for (int s0 = 0; s0 < kTile && tt + s0 < sg.t1; s0 += kSplitBoxRows)
#pragma unroll
            for (int bx = 0; bx < Gm::kBoxes; ++bx) {
              tma_prefetch_3d(&kmap, bx * 64, base + tt + s0, pair);
              tma_prefetch_3d(&vmap, bx * 64, base + tt + s0, pair);
            }
      } while (left > 0 && next_seg(prefix, Hkv, r1, sg));
    }
  }
  pdl_wait_prior_grid();
  if (clamped) atomicOr(hdr + kHdrError, kErrLenClamped);
  // the mark of a piece done in this launch: the launch's epoch with the top bit set
  // (no sequence offset, and no partial of a finite attention, has that bit pattern)
  const uint32_t mark =
      kFused ? 0x80000000u | ((*reinterpret_cast<volatile uint32_t *>(hdr + kHdrEpoch) + 1u) &
                              0x7fffffffu)
             : 0u;
  if (blockIdx.x == 0 && tid == 0) hdr[kHdrDirect] = out_direct != nullptr;
  if (blockIdx.x == 0) {  // the merge pass reads the sequence offsets from here
    int *wp = reinterpret_cast<int *>(workspace + ws_prefix_offset(gridDim.x, B, Hkv, G, D));
    for (int b = tid; b <= B; b += kNT) wp[b] = prefix[b];
  }

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      const uint32_t q_bytes = (uint32_t)(G * D * 2);
      uint32_t it = 0;
      int last_n[kMaxStages];
#pragma unroll
      for (int s = 0; s < kMaxStages; ++s) last_n[s] = -1;
      // claim a stage for tile number `it`; false once the pipeline has given up
      auto acquire = [&](int &st) -> bool {
        st = (int)(it % stages);
        const int n = (int)(it / stages);
        if (s_abort) return false;
        if (n > 0 && !mbar_wait_bounded(bar_empty + 8 * st, (n - 1) & 1)) {
          atomicOr(hdr + kHdrError, kErrWaitTimeout);
          s_abort = 1;
          return false;
        }
        last_n[st] = n;
        return true;
      };

      long long piece = (long long)blockIdx.x * kPiecesPerBlock;  // this CTA's large piece
      long long next = -1;
      const bool has_small = sched.big < sched.blk;
      while (true) {
        const long long r0 = sched.start(piece), r1 = sched.start(piece + 1);
        if (piece < 0 || (piece % kPiecesPerBlock != 0 && r0 >= total)) break;
        if (next == -1) {
          const long long k = has_small ? (long long)atomicAdd(hdr + kHdrNextPiece, 1u) : -1;
          next = (k >= 0 && k < (long long)gridDim.x * kSmallPiecesPerBlock)
                     ? PieceSched::small_piece(k) : -2;
        }
        bool listed = false;
        if (kFused && r0 < r1 && s_npieces < kPieceList) {
          s_pieces[s_npieces] = (int)piece;
          s_npieces = s_npieces + 1;
          listed = true;
        }
        if (r0 < r1 && !s_abort) {
          Seg sg = first_seg(prefix, B, Hkv, r0, r1);
          do {
            const int pair = sg.b * Hkv + sg.g;
            const int L = seq_len(prefix, sg.b);
            // token 0 of the run's coordinates is cache row `base`: the window's first row
            int Lfull = lens[sg.b];
            Lfull = Lfull < 0 ? 0 : (Lfull > T_cap ? T_cap : Lfull);
            const int base = Lfull - L;
            for (int tt = sg.t0; tt < sg.t1; tt += kTile) {
              const int rows = min(kTile, sg.t1 - tt);
              const int nload = rows == kTile ? kTile : (rows + kSubRows - 1) & ~(kSubRows - 1);
              const bool first = tt == sg.t0;
              int st;
              if (!acquire(st)) break;
              TileMeta &m = meta[st];
              m.b = sg.b; m.g = sg.g; m.tok0 = tt; m.tok_end = sg.t1; m.L = L; m.nload = nload;
              m.slot = (int)(piece + pair);
              m.piece = (int)piece;
              const bool last_tile = tt + kTile >= sg.t1;
              m.flags = (first ? kFirst : 0u) | (last_tile ? kLast : 0u) |
                        (!listed && last_tile && sg.r + (sg.t1 - sg.t0) >= r1 ? kPieceEnd : 0u);
              const uint32_t full = bar_full + 8 * st;
              mbar_arrive_expect_tx(full, (uint32_t)(2 * nload * 128 * Gm::kBoxes) +
                                              (first ? q_bytes : 0u));
              const uint32_t kt = s_base + st * Gm::kStageBytes;
              const uint32_t vt = kt + Gm::kTileBytes;
              // whole 64-row boxes first, then 8-row boxes up to nload
              int s0 = 0;
              for (; s0 + kSplitBoxRows <= nload; s0 += kSplitBoxRows) {
#pragma unroll
                for (int bx = 0; bx < Gm::kBoxes; ++bx) {
                  const uint32_t off = bx * Gm::kBoxBytes + s0 * 128;
                  tma_load_3d(kt + off, &kmap, bx * 64, base + tt + s0, pair, full, policy);
                  tma_load_3d(vt + off, &vmap, bx * 64, base + tt + s0, pair, full, policy);
                }
              }
              for (; s0 < nload; s0 += kSubRows) {
#pragma unroll
                for (int bx = 0; bx < Gm::kBoxes; ++bx) {
                  const uint32_t off = bx * Gm::kBoxBytes + s0 * 128;
                  tma_load_3d(kt + off, &kmap8, bx * 64, base + tt + s0, pair, full, policy);
                  tma_load_3d(vt + off, &vmap8, bx * 64, base + tt + s0, pair, full, policy);
                }
              }
              if (first)
                bulk_load(s_base + lay.q_off + st * lay.q_stride,
                          q + ((size_t)sg.b * Hq + (size_t)sg.g * G) * D, q_bytes, full);
              ++it;
            }
          } while (!s_abort && next_seg(prefix, Hkv, r1, sg));
        }
        piece = next;  // -2: no small piece left
        next = -1;
      }
      // tell the consumers there is nothing more
      int st;
      if (acquire(st)) {
        meta[st].flags = kEnd;
        mbar_arrive(bar_full + 8 * st);
      }
      // the last CTA to finish claiming resets the claim counters for the next launch
      __threadfence();
      if (atomicAdd(hdr + kHdrDone, 1u) == gridDim.x - 1) {
        atomicExch(hdr + kHdrNextPiece, 0u);
        atomicExch(hdr + kHdrDone, 0u);
      }
      // no copy may still be in flight into this CTA's shared memory when it exits
      for (int s = 0; s < stages; ++s)
        if (last_n[s] >= 0) mbar_wait_bounded(bar_full + 8 * s, last_n[s] & 1);
    }
    if constexpr (kFused) {
      __syncwarp();
      merge_phase<D>(hdr, workspace, prefix, sched, scratch, out_direct, B, Hq, Hkv, G,
                     merge_wph, mark, s_pieces, s_npieces);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int row0 = 16 * warp;  // first tile row of this warp
  const int gid = lane >> 2, tig = lane & 3;
  const float NEG_INF = -INFINITY;
  float *o_ws = reinterpret_cast<float *>(workspace + kWsHeaderBytes);
  float *lse_ws = reinterpret_cast<float *>(workspace + ws_lse_offset(gridDim.x, B, Hkv, G, D));
  const int ws_stride = lay.warp_scratch;

  uint32_t qf[KS][2];
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  float o[MT][4];
  uint32_t fin_n = 0;
  uint32_t runs_done = 0;  // run ends whose combine this warp has finished
  bool ok = true;
  int run_t0 = 0;  // first token of the current run

  // rendezvous of the consumer warps, bounded
  auto fin_sync = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_fin);
    if (!mbar_wait_bounded(bar_fin, fin_n & 1)) {
      if (lane == 0) atomicOr(hdr + kHdrError, kErrWaitTimeout);
      s_abort = 1;
      ok = false;
    }
    ++fin_n;
  };

  for (uint32_t it = 0; ok; ++it) {
    const int st = (int)(it % stages);
    const int n = (int)(it / stages);
    if (!mbar_wait_bounded(bar_full + 8 * st, n & 1)) {
      if (lane == 0) atomicOr(hdr + kHdrError, kErrWaitTimeout);
      s_abort = 1;
      break;
    }
    const TileMeta m = meta[st];
    if (m.flags & kEnd) break;
    if (m.flags & kFirst) {
      run_t0 = m.tok0;
      // Q^T operand (k = head dim, n = query head of the group); heads >= G are zero.
      const bool hv = gid < G;
      const uint32_t qa = s_base + lay.q_off + st * lay.q_stride + (hv ? gid : 0) * D * 2;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a, b;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a) : "r"(qa + (16 * ks + 2 * tig) * 2));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b) : "r"(qa + (16 * ks + 8 + 2 * tig) * 2));
        qf[ks][0] = hv ? a : 0u;
        qf[ks][1] = hv ? b : 0u;
      }
      m0 = NEG_INF; m1 = NEG_INF; l0 = 0.f; l1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }
    const int tok0 = m.tok0 + row0;  // token of this warp's first row
    if (tok0 < m.tok_end) {
      const uint32_t kt = s_base + st * Gm::kStageBytes;
      const uint32_t vt = kt + Gm::kTileBytes;
      // rows past the loaded ones, or at or past the run's end, may hold stale data or
      // NaN (past the sequence's length, or a slot another writer may be filling while
      // this run reads past its end): zero their V (their scores are masked by index
      // below)
      const int zero_from = min(m.nload, m.tok_end - m.tok0);
      if (row0 + 16 > zero_from) {
        const int rlo = max(zero_from, row0);
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
      const bool va = tok0 + gid < m.tok_end, vb = tok0 + gid + 8 < m.tok_end;
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

    if (m.flags & kLast) {
      // ---- combine the warps' states of this run into one partial
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      // the previous combine's reads of the scratch are over (a wait that has almost
      // always completed by now)
      if (runs_done > 0 && !mbar_wait_bounded(bar_free, (runs_done - 1) & 1)) {
        if (lane == 0) atomicOr(hdr + kHdrError, kErrWaitTimeout);
        s_abort = 1;
        ok = false;
        break;
      }
      {
        float *sw = scratch + warp * ws_stride;
        float *sm = sw + G * Gm::kOStride;
        float *sl = sm + G;
        const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int d = 16 * mt + gid;
          if (h0 < G) {
            sw[h0 * Gm::kOStride + d] = o[mt][0];
            sw[h0 * Gm::kOStride + d + 8] = o[mt][2];
          }
          if (h1 < G) {
            sw[h1 * Gm::kOStride + d] = o[mt][1];
            sw[h1 * Gm::kOStride + d + 8] = o[mt][3];
          }
        }
        if (gid == 0) {
          if (h0 < G) { sm[h0] = m0; sl[h0] = l0; }
          if (h1 < G) { sm[h1] = m1; sl[h1] = l1; }
        }
      }
      fin_sync();
      const size_t slot = (size_t)m.slot;
      // a run that is the whole (b, g) pair is the final answer: write it as bf16
      __nv_bfloat16 *od = (out_direct != nullptr && run_t0 == 0 && m.tok_end == m.L)
                              ? out_direct + ((size_t)m.b * Hq + (size_t)m.g * G) * D
                              : nullptr;
      if (ok) {
        // each thread four consecutive elements of one head, forming that head's weights
        // itself (warp w's share 2^(m_w - M) / sum), so the sums follow the first
        // rendezvous directly; 16-byte reads of the warps' states and 16-byte writes
        float *op = o_ws + slot * G * D;
        constexpr int Q = D / 4;  // quads per head
        for (int qd = tid; qd < G * Q; qd += kConsumerThreads) {
          const int h = qd / Q, d = (qd - h * Q) * 4;
          const float *sm_h = scratch + G * Gm::kOStride + h;  // warp w's m at w * ws_stride
          float M = NEG_INF;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_h[w * ws_stride]);
          float f[kConsumerWarps];
          float wsum = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = sm_h[w * ws_stride];
            f[w] = (mw == NEG_INF) ? 0.f : exp2f(mw - M);
            wsum += f[w] * sm_h[w * ws_stride + G];
          }
          const float inv = 1.f / wsum;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = f[w] * inv;
            const float4 v = *reinterpret_cast<const float4 *>(scratch + w * ws_stride +
                                                               h * Gm::kOStride + d);
            acc.x = fmaf(wt, v.x, acc.x);
            acc.y = fmaf(wt, v.y, acc.y);
            acc.z = fmaf(wt, v.z, acc.z);
            acc.w = fmaf(wt, v.w, acc.w);
          }
          if (od != nullptr) {
            *reinterpret_cast<uint2 *>(od + h * D + d) =
                make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
          } else {
            *reinterpret_cast<float4 *>(op + h * D + d) = acc;
            if (d == 0) lse_ws[slot * G + h] = M + log2f(wsum);
          }
        }
        // release the scratch without waiting for the other warps: the next combine
        // waits for this release before it writes
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_free);
        ++runs_done;
        // a run that closes an unlisted piece marks it done, after every consumer's
        // stores of it (the rendezvous)
        if (kFused && (m.flags & kPieceEnd)) {
          fin_sync();
          if (tid == 0) {
            fence_acq_rel_gpu();
            st_release_gpu(reinterpret_cast<uint32_t *>(
                               workspace + ws_flags_offset(gridDim.x, B, Hkv, G, D)) + m.piece,
                           mark);
          }
        }
      }
    }
  }
  if constexpr (kFused)
    merge_phase<D>(hdr, workspace, prefix, sched, scratch, out_direct, B, Hq, Hkv, G, merge_wph,
                   mark, s_pieces, s_npieces);
}

// Merge: one group of `wph` warps per query head (8 warps per CTA, or one head of
// wph > 8 warps per CTA).
// Each warp takes every wph-th partial of its head's run of pieces: a first pass
// finds its largest lse, a second accumulates 2^(lse - M) o with independent loads;
// the group's warps are then combined through shared memory.
template <int D>
__global__ void __launch_bounds__(1024) split_merge_kernel(const uint8_t *__restrict__ workspace,
                                                           __nv_bfloat16 *__restrict__ out, int B,
                                                           int Hq, int Hkv, int num_parts,
                                                           int wph) {
  constexpr int E = D / 32;  // floats per lane
  __shared__ float s_m[32], s_w[32];
  __shared__ float s_acc[32][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hpc = (blockDim.x >> 5) / wph;  // heads per CTA
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int hs = warp / wph, sub = warp - hs * wph;
  const int b = blockIdx.y;
  const int h = blockIdx.x * hpc + hs;
  const int G = Hq / Hkv;
  const int *prefix =
      reinterpret_cast<const int *>(workspace + ws_prefix_offset(num_parts, B, Hkv, G, D));
  const float *o_ws = reinterpret_cast<const float *>(workspace + kWsHeaderBytes);
  const float *lse_ws =
      reinterpret_cast<const float *>(workspace + ws_lse_offset(num_parts, B, Hkv, G, D));
  const int pre = prefix[b], Lb = prefix[b + 1] - pre;
  const PieceSched sched = PieceSched::make((long long)Hkv * prefix[B], num_parts);
  const bool direct = reinterpret_cast<const uint32_t *>(workspace)[kHdrDirect] != 0;
  // a head whose pair fell in a single piece was written by the split pass already
  bool done = false;
  if (direct && h < Hq && Lb > 0) {
    const long long start = (long long)Hkv * pre + (long long)(h / G) * Lb;
    done = sched.piece_of(start) == sched.piece_of(start + Lb - 1);
  }

  float M = -INFINITY, wsum = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  if (h < Hq && Lb > 0 && !done) {
    const int g = h / G, hh = h - g * G;
    const long long pair = (long long)b * Hkv + g;
    const long long start = (long long)Hkv * pre + (long long)g * Lb;
    // pieces [c0, c1] cover the pair; the empty ones (the small pieces of blocks too
    // short to split) wrote nothing and are skipped
    const long long c0 = sched.piece_of(start), c1 = sched.piece_of(start + Lb - 1);
    for (long long c = c0 + sub + (long long)wph * lane; c <= c1; c += 32ll * wph)
      if (!sched.empty(c)) M = fmaxf(M, lse_ws[(c + pair) * G + hh]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M > -INFINITY) {
      auto add = [&](long long c, float lse, const float *op) {
        const float w = exp2f(lse - M);
        wsum += w;
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4 *>(op);
          acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2 *>(op);
          acc[0] += w * v.x; acc[1] += w * v.y;
        }
      };
      long long c = c0 + sub;
      for (; c + 3ll * wph <= c1; c += 4ll * wph) {
        float l4[4];
        const float *p4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long cu = c + (long long)u * wph;
          const long long slot = cu + pair;
          l4[u] = sched.empty(cu) ? -INFINITY : lse_ws[slot * G + hh];
          p4[u] = o_ws + (slot * G + hh) * D + lane * E;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (l4[u] > -INFINITY) add(c + u * wph, l4[u], p4[u]);
      }
      for (; c <= c1; c += wph) {
        if (sched.empty(c)) continue;
        const long long slot = c + pair;
        add(c, lse_ws[slot * G + hh], o_ws + (slot * G + hh) * D + lane * E);
      }
    }
  }
  if (lane == 0) { s_m[warp] = M; s_w[warp] = wsum; }
#pragma unroll
  for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
  __syncthreads();
  if (sub != 0 || h >= Hq || done) return;
  float Mh = -INFINITY;
  for (int w = 0; w < wph; ++w) Mh = fmaxf(Mh, s_m[hs * wph + w]);
  float tot = 0.f, r[E];
#pragma unroll
  for (int e = 0; e < E; ++e) r[e] = 0.f;
  if (Mh > -INFINITY) {
    for (int w = 0; w < wph; ++w) {
      const int ww = hs * wph + w;
      const float f = s_m[ww] == -INFINITY ? 0.f : exp2f(s_m[ww] - Mh);
      tot += f * s_w[ww];
#pragma unroll
      for (int e = 0; e < E; ++e) r[e] += f * s_acc[ww][lane * E + e];
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  __nv_bfloat16 *orow = out + ((size_t)b * Hq + h) * D + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(orow) = make_uint2(pack_bf16x2(r[0] * inv, r[1] * inv),
                                                  pack_bf16x2(r[2] * inv, r[3] * inv));
  } else {
    *reinterpret_cast<uint32_t *>(orow) = pack_bf16x2(r[0] * inv, r[1] * inv);
  }
}

// Dynamic shared memory a split kernel instance may use on `device`: the opt-in
// per-block limit minus the kernel's static shared memory. Cached per device.
template <int D, int kMode>
int split_smem_cap(int device) {
  static int cap[64] = {0};
  if (device < 0 || device >= 64) return 0;
  if (cap[device] == 0) {
    int optin = 0;
    cudaFuncAttributes attr{};
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess ||
        cudaFuncGetAttributes(&attr, gqa_split_kernel<D, kMode>) != cudaSuccess)
      return 0;
    cap[device] = optin - (int)attr.sharedSizeBytes;
  }
  return cap[device];
}

template <int D, int kMode>
cudaError_t ensure_split_attr(int device) {
  static int done[64] = {0};
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gqa_split_kernel<D, kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       split_smem_cap<D, kMode>(device));
  if (e == cudaSuccess) done[device] = 1;
  return e;
}

// The one-launch attention: a cooperative launch (every CTA resident at once, which
// the grid barrier needs) that may also start early behind the previous kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Warps per query head for merging pairs of up to max_len rows (a pair of L rows meets
// about kPiecesPerBlock * L / blk pieces); any value gives the same result.
int merge_warps_per_head(int B, int Hkv, int max_len, int num_parts, int cap) {
  const long long rows = (long long)B * Hkv * (long long)max_len;
  const long long blk = (rows + num_parts - 1) / num_parts;
  const long long est = blk > 0 ? (long long)kPiecesPerBlock * max_len / blk + 2 : 1;
  int wph = 1;
  while (wph < cap && wph * 8 < est) wph *= 2;
  return wph;
}

}  // namespace

int split_stages(int D, int G, int B, int device) {
  // the same layout in both modes: the smaller room either leaves
  const int cap = D == 128 ? min(split_smem_cap<128, 0>(device), split_smem_cap<128, 1>(device))
                           : min(split_smem_cap<64, 0>(device), split_smem_cap<64, 1>(device));
  for (int s = kSplitMaxStages; s >= 2; --s)
    if (split_layout(D, G, B, s).bytes <= cap) return s;
  return 0;
}

size_t split_smem_bytes(int D, int G, int B, int stages) {
  return (size_t)split_layout(D, G, B, stages).bytes;
}

bool split_fused_fits(int num_parts, int device) {
  int sms = 0, coop = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess)
    return false;
  return coop != 0 && num_parts >= 1 && num_parts <= sms;  // one CTA per SM
}

cudaError_t launch_gqa_split(const CUtensorMap &kmap, const CUtensorMap &vmap,
                             const CUtensorMap &kmap8, const CUtensorMap &vmap8, const void *q,
                             const int32_t *lens, int B, int Hq, int Hkv, int D, int T_cap,
                             float scale_log2, int num_parts, void *workspace, void *out_direct,
                             int window, cudaStream_t stream, bool fused, int max_len) {
  auto *odp = static_cast<__nv_bfloat16 *>(out_direct);
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const int G = Hq / Hkv;
  const int stages = split_stages(D, G, B, device);
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = split_smem_bytes(D, G, B, stages);
  auto *qp = static_cast<const __nv_bfloat16 *>(q);
  auto *ws = static_cast<uint8_t *>(workspace);
  if (fused && odp == nullptr) return cudaErrorInvalidValue;
  const int wph = merge_warps_per_head(B, Hkv, max_len, num_parts, kConsumerWarps);
  auto go = [&](auto kernel, bool coop) {
    return coop ? launch_coop_pdl(kernel, num_parts, kThreads, smem, stream, kmap, vmap, kmap8,
                                  vmap8, qp, lens, B, Hq, Hkv, T_cap, scale_log2, stages, ws,
                                  odp, window, wph)
                : launch_pdl(kernel, num_parts, kThreads, smem, stream, kmap, vmap, kmap8,
                             vmap8, qp, lens, B, Hq, Hkv, T_cap, scale_log2, stages, ws, odp,
                             window, 1);
  };
  if (D == 128) {
    if (fused) {
      if ((e = ensure_split_attr<128, 1>(device)) != cudaSuccess) return e;
      e = go(gqa_split_kernel<128, 1>, true);
    } else {
      if ((e = ensure_split_attr<128, 0>(device)) != cudaSuccess) return e;
      e = go(gqa_split_kernel<128, 0>, false);
    }
  } else {
    if (fused) {
      if ((e = ensure_split_attr<64, 1>(device)) != cudaSuccess) return e;
      e = go(gqa_split_kernel<64, 1>, true);
    } else {
      if ((e = ensure_split_attr<64, 0>(device)) != cudaSuccess) return e;
      e = go(gqa_split_kernel<64, 0>, false);
    }
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_split_merge(const void *workspace, void *out, int B, int Hq, int Hkv, int D,
                               int max_len, int num_parts, cudaStream_t stream) {
  auto *ws = static_cast<const uint8_t *>(workspace);
  auto *op = static_cast<__nv_bfloat16 *>(out);
  const int wph = merge_warps_per_head(B, Hkv, max_len, num_parts, 32);
  const int threads = wph <= 8 ? 256 : 32 * wph;
  const int hpc = (threads / 32) / wph;
  const dim3 grid((unsigned)((Hq + hpc - 1) / hpc), (unsigned)B);
  cudaError_t e;
  if (D == 128)
    e = launch_pdl(split_merge_kernel<128>, grid, threads, 0, stream, ws, op, B, Hq, Hkv,
                   num_parts, wph);
  else
    e = launch_pdl(split_merge_kernel<64>, grid, threads, 0, stream, ws, op, B, Hq, Hkv, num_parts,
                   wph);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace decattn
