// Device helpers shared by the sm_103a kernels of the decode-step attention block:
// bf16 packing, warp reductions, mbarrier / bulk-tensor (TMA) / ldmatrix / movmatrix /
// mma wrappers written as inline PTX.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace decattn {

// ------------------------------------------------------------ scheduling ---
// Geometry of the split pass of the attention.
constexpr int kSplitTile = 128;    // tokens per pipeline stage of the split pass
constexpr int kSplitBoxRows = 64;  // tokens per full bulk-tensor box (two per tile)
constexpr int kSplitMaxB = 8192;   // largest batch the split pass keeps prefix sums for
constexpr int kSplitMaxG = 8;      // largest query-head group per KV head
constexpr int kSplitMaxStages = 8; // most pipeline stages the split pass uses

// Smallest number of (sequence, KV head, token) rows one split-pass CTA takes.
constexpr int kMinRowsPerPart = 64;
// Wall-clock bound of one pipeline wait before the kernel gives up (ns). A healthy
// wait lasts microseconds; a phase that never completes is reported, not hung on.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Bits of the device error word (mirrors DEC_DEVERR_* of the public header).
constexpr uint32_t kErrLenClamped = 0x1u;
constexpr uint32_t kErrPosSkipped = 0x2u;
constexpr uint32_t kErrWaitTimeout = 0x4u;

// How the split pass cuts the stream of (sequence, KV head, token) rows into pieces.
// The stream is split into P equal blocks of `blk` rows, one per CTA. When a block is
// large enough, its first 4/5 is the CTA's own piece (taken statically) and the rest
// is cut into 4 small pieces that any CTA claims from a counter once it is done, so
// the SMs that get more bandwidth do more of the work and all finish together;
// smaller blocks are one piece each. Piece 5c is block c's large piece and 5c+1+j
// its j-th small piece, so pieces are numbered in stream order, their boundaries are
// a closed form of the index, and the merge finds a pair's pieces without any record
// of who ran them: results do not depend on the claim order.
// 4 small pieces of a fifth of a block: fewer runs (each ends in a combine of the
// warps' states) than finer cuts, fine enough to even out the SMs' bandwidth (tuned
// on the batched, long-context and serving workloads).
constexpr int kSmallPiecesPerBlock = 4;
constexpr long long kBigPermille = 800;  // share of a block its own CTA takes
constexpr int kPiecesPerBlock = 1 + kSmallPiecesPerBlock;
constexpr long long kMinSplitBlockRows = 4096;  // smaller blocks are not split

struct PieceSched {
  long long total, blk, big, cs;
  int P;

  __host__ __device__ static PieceSched make(long long total_rows, int num_parts) {
    PieceSched s;
    s.total = total_rows;
    s.P = num_parts;
    long long blk = (total_rows + num_parts - 1) / num_parts;
    s.blk = blk < kMinRowsPerPart ? (long long)kMinRowsPerPart : blk;
    if (s.blk >= kMinSplitBlockRows) {
      s.big = s.blk * kBigPermille / 1000;
      s.cs = (s.blk - s.big + kSmallPiecesPerBlock - 1) / kSmallPiecesPerBlock;
    } else {
      s.big = s.blk;
      s.cs = 1;
    }
    return s;
  }
  // first row of piece i (the end of the stream for i past the last piece)
  __host__ __device__ long long start(long long i) const {
    const long long c = i / kPiecesPerBlock, j = i - c * kPiecesPerBlock;
    const long long bs = c * blk;
    long long r = j == 0 ? bs : bs + big + (j - 1) * cs;
    const long long be = bs + blk;
    r = r < be ? r : be;
    return r < total ? r : total;
  }
  __host__ __device__ long long piece_of(long long row) const {
    const long long c = row / blk, off = row - c * blk;
    return off < big ? c * kPiecesPerBlock : c * kPiecesPerBlock + 1 + (off - big) / cs;
  }
  __host__ __device__ bool empty(long long i) const { return start(i) >= start(i + 1); }
  // The same in 32-bit arithmetic, for streams of fewer than 2^31 rows (the launch
  // checks B * Hkv * T_cap < 2^31): a fraction of the cost of 64-bit division.
  __device__ unsigned start32(unsigned i) const {
    const unsigned c = i / kPiecesPerBlock, j = i - c * kPiecesPerBlock;
    const unsigned bs = c * (unsigned)blk;
    unsigned r = j == 0 ? bs : bs + (unsigned)big + (j - 1) * (unsigned)cs;
    const unsigned be = bs + (unsigned)blk;
    r = r < be ? r : be;
    return r < (unsigned)total ? r : (unsigned)total;
  }
  __device__ unsigned piece_of32(unsigned row) const {
    const unsigned c = row / (unsigned)blk, off = row - c * (unsigned)blk;
    return off < (unsigned)big ? c * kPiecesPerBlock
                               : c * kPiecesPerBlock + 1 + (off - (unsigned)big) / (unsigned)cs;
  }
  __device__ bool empty32(unsigned i) const { return start32(i) >= start32(i + 1); }
  // index of the k-th claimable small piece
  __host__ __device__ static long long small_piece(long long k) {
    return (k / kSmallPiecesPerBlock) * kPiecesPerBlock + 1 + k % kSmallPiecesPerBlock;
  }
};

// Upper bound of the piece count for any number of rows.
__host__ __device__ inline long long max_pieces(int num_parts) {
  return (long long)num_parts * kPiecesPerBlock;
}

// Attention workspace layout: a 256-byte header, the o partials fp32 [S][G][D], the
// lse partials fp32 [S][G], then the sequence offsets int32 [B+1] (exclusive prefix
// sums of the clamped lengths, written by the split pass for the merge), with
// S = max_pieces(P) + B*Hkv partial slots.
constexpr size_t kWsHeaderBytes = 256;
__host__ __device__ inline size_t ws_slots(int P, int B, int Hkv) {
  return (size_t)max_pieces(P) + (size_t)B * Hkv;
}
__host__ __device__ inline size_t ws_lse_offset(int P, int B, int Hkv, int G, int D) {
  return kWsHeaderBytes + ws_slots(P, B, Hkv) * G * D * 4;
}
__host__ __device__ inline size_t ws_prefix_offset(int P, int B, int Hkv, int G, int D) {
  return (ws_lse_offset(P, B, Hkv, G, D) + ws_slots(P, B, Hkv) * G * 4 + 15) & ~(size_t)15;
}
// then one completion word per piece (uint32 [5P]): the one-launch attention marks a
// piece done with the launch's epoch, and merges a head once all its pieces are marked
__host__ __device__ inline size_t ws_flags_offset(int P, int B, int Hkv, int G, int D) {
  return (ws_prefix_offset(P, B, Hkv, G, D) + (size_t)(B + 1) * 4 + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t ws_total_bytes(int P, int B, int Hkv, int G, int D) {
  return (ws_flags_offset(P, B, Hkv, G, D) + (size_t)max_pieces(P) * 4 + 255) & ~(size_t)255;
}

// ------------------------------------------------------------------ bf16 ---
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// ----------------------------------------------------------------- warps ---
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------- programmatic dependent launch ---
// Kernels are launched so that the next kernel on the stream may be scheduled before
// they finish. Each kernel lets its dependent launch early and, before touching any
// input in global memory, waits until the previous grid on the stream has completed
// and its writes are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// -------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; false once kWaitLimitNs of
// wall-clock time has passed (each try_wait may itself suspend the thread for a
// while, so the bound is on time, not on the number of tries).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// ------------------------------------------------------------------- TMA ---
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 3-D tiled bulk-tensor prefetch of a box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const void *tmap, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// 3-D tiled bulk-tensor load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int c0, int c1, int c2,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ------------------------------------------------------- ldmatrix / mma ---
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace decattn
