// The C ABI of libdecattn.so (declared in include/decattn.h): host-side argument
// checks, launch geometry, bulk-tensor descriptors of the KV cache, and launches.
// Nothing here allocates, frees or synchronises.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>

#include "decattn.h"
#include "dec_device.cuh"
#include "dec_launch.h"
#include "rope_angles.cuh"

namespace {

using namespace decattn;

thread_local char g_last_error[256] = "";

dec_status fail(dec_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

dec_status ok() {
  g_last_error[0] = '\0';
  return DEC_OK;
}

dec_status cuda_fail(cudaError_t e, const char *where) {
  return fail(DEC_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(dec_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Where the kernels may find a buffer. Plain loads and stores reach device memory and
// page-locked host memory that is mapped into the device's address space at the same
// address (unified addressing); bulk-tensor and bulk copies are only ever given device
// memory. Any other pointer would fault the GPU, so it is refused before a launch.
dec_status where_ok(const void *p, const char *name, bool host_ok) {
  if (p == nullptr) return DEC_OK;
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return cuda_fail(e, name);
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return DEC_OK;
  if (host_ok && a.type == cudaMemoryTypeHost && a.devicePointer == p) return DEC_OK;
  return fail(DEC_ERR_INVALID_ARG, host_ok ? "%s is neither device memory nor page-locked host "
                                             "memory mapped at the same address"
                                           : "%s must be device memory",
              name);
}

struct Where {
  const void *p;
  const char *name;
  bool host_ok;
};

dec_status where_all(std::initializer_list<Where> list) {
  for (const Where &w : list) {
    const dec_status st = where_ok(w.p, w.name, w.host_ok);
    if (st != DEC_OK) return st;
  }
  return DEC_OK;
}

// The RoPE frequency table of a call: the caller's D/2 values (host memory, read now,
// each in [0, 1]) or, without one, theta^(-2i/D).
dec_status rope_table(int D, float rope_theta, const double *inv_freq, InvFreq *out) {
  if (inv_freq == nullptr) {
    if (!(rope_theta > 0.f) || std::isinf(rope_theta))
      return fail(DEC_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
    *out = make_inv_freq(D, (double)rope_theta);
    return DEC_OK;
  }
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, inv_freq);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return cuda_fail(e, "inv_freq");
  }
  if (a.type == cudaMemoryTypeDevice)
    return fail(DEC_ERR_INVALID_ARG, "inv_freq must be host memory (the host reads it)");
  for (int i = 0; i < D / 2; ++i) {
    const double v = inv_freq[i];
    if (!(v >= 0.0 && v <= 1.0))
      return fail(DEC_ERR_INVALID_ARG, "inv_freq[%d] = %g is outside [0, 1]", i, v);
    out->v[i] = v;
  }
  return DEC_OK;
}

// Per-device cache of the SM count.
std::atomic<int> g_sm_count[64];

int sm_count(int device) {
  if (device < 0 || device >= 64) return 1;
  int n = g_sm_count[device].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
    n = 1;
  g_sm_count[device].store(n, std::memory_order_relaxed);
  return n;
}

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) d = 0;
  return d;
}

int sm_count_of_current() { return sm_count(current_device()); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A [B*Hkv, T_cap, D] bf16 cache as a 3-D tensor; boxes of 64 dims x box_rows tokens
// x 1 pair, 128-byte swizzle. Rows past T_cap read as zeros.
dec_status encode_cache_map(CUtensorMap *map, const void *cache, int B, int Hkv, int D,
                            int T_cap, int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return fail(DEC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T_cap, (cuuint64_t)B * (cuuint64_t)Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T_cap * (cuuint64_t)D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(cache), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DEC_OK;
}

dec_status check_attn_shape(int B, int Hq, int Hkv, int D, int T_cap, int max_len) {
  if (B < 0) return fail(DEC_ERR_INVALID_ARG, "B = %d < 0", B);
  if (Hq <= 0 || Hkv <= 0) return fail(DEC_ERR_INVALID_ARG, "head counts must be positive");
  if (Hq % Hkv != 0) return fail(DEC_ERR_INVALID_ARG, "Hq = %d is not a multiple of Hkv = %d", Hq, Hkv);
  if (D != 64 && D != 128) return fail(DEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (Hq / Hkv > kSplitMaxG)
    return fail(DEC_ERR_UNSUPPORTED, "query heads per KV head %d > %d", Hq / Hkv, kSplitMaxG);
  if (T_cap <= 0) return fail(DEC_ERR_INVALID_ARG, "T_cap = %d must be positive", T_cap);
  if (max_len < 0 || max_len > T_cap)
    return fail(DEC_ERR_INVALID_ARG, "max_len = %d outside [0, T_cap = %d]", max_len, T_cap);
  if (B > kSplitMaxB) return fail(DEC_ERR_UNSUPPORTED, "B = %d > %d", B, kSplitMaxB);
  if ((long long)B * Hkv * (long long)T_cap >= (1ll << 31))
    return fail(DEC_ERR_UNSUPPORTED, "B * Hkv * T_cap must stay below 2^31 rows");
  return DEC_OK;
}

int resolve_parts(int num_parts, int B, int Hkv, int D, int max_len) {
  if (num_parts > 0) return num_parts;
  return dec_attn_default_parts(B, Hkv, D, max_len);
}

size_t workspace_bytes(int B, int Hq, int Hkv, int D, int parts) {
  return ws_total_bytes(parts, B, Hkv, Hq / Hkv, D);
}

}  // namespace

namespace decattn {
dec_status record_error(dec_status status, const char *message) {
  return fail(status, "%s", message);
}
}  // namespace decattn

extern "C" {

const char *dec_status_string(dec_status s) {
  switch (s) {
    case DEC_OK: return "ok";
    case DEC_ERR_INVALID_ARG: return "invalid argument";
    case DEC_ERR_UNSUPPORTED: return "unsupported shape";
    case DEC_ERR_WORKSPACE: return "workspace too small";
    case DEC_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char *dec_last_error(void) { return g_last_error; }

int dec_version(void) { return 100; }

dec_status dec_rmsnorm_residual(const void *x, void *residual, const void *weight, void *y,
                                int B, int hidden, float eps, dec_stream_t stream) {
  if (B < 0) return fail(DEC_ERR_INVALID_ARG, "B = %d < 0", B);
  if (hidden < 8 || hidden > 16384 || hidden % 8 != 0)
    return fail(DEC_ERR_UNSUPPORTED, "hidden = %d (need a multiple of 8 in [8, 16384])", hidden);
  if (!(eps >= 0.f)) return fail(DEC_ERR_INVALID_ARG, "eps must be >= 0");
  if (B == 0) return ok();
  if (!x || !weight || !y) return fail(DEC_ERR_INVALID_ARG, "x, weight and y must be non-null");
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y) || (residual && !aligned16(residual)))
    return fail(DEC_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (y == x || (residual != nullptr && y == residual))
    return fail(DEC_ERR_INVALID_ARG, "y may not alias x or residual");
  dec_status st = where_all({{x, "x", true}, {residual, "residual", true}, {weight, "weight", true},
                             {y, "y", true}});
  if (st != DEC_OK) return st;
  cudaError_t e = launch_rmsnorm_residual(x, residual, weight, y, B, hidden, eps, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm_residual launch");
  return ok();
}

}  // extern "C"

namespace {
dec_status qknorm_rope_impl(const void *q_in, void *q_out, const void *k_new, const void *v_new,
                            const void *q_norm_w, const void *k_norm_w, void *k_cache,
                            void *v_cache, const int32_t *pos, int B, int Hq, int Hkv, int D,
                            int T_cap, float rope_theta, dec_rope_layout layout,
                            const double *inv_freq, float eps, uint32_t *error_word,
                            dec_stream_t stream) {
  if (B < 0) return fail(DEC_ERR_INVALID_ARG, "B = %d < 0", B);
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(DEC_ERR_INVALID_ARG, "need Hq, Hkv > 0 and Hq %% Hkv == 0");
  if (D != 64 && D != 128) return fail(DEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (T_cap <= 0) return fail(DEC_ERR_INVALID_ARG, "T_cap = %d must be positive", T_cap);
  InvFreq inv;
  dec_status st = rope_table(D, rope_theta, inv_freq, &inv);
  if (st != DEC_OK) return st;
  if (layout != DEC_ROPE_NEOX && layout != DEC_ROPE_INTERLEAVED)
    return fail(DEC_ERR_INVALID_ARG, "unknown rope layout %d", (int)layout);
  if (!(eps >= 0.f)) return fail(DEC_ERR_INVALID_ARG, "eps must be >= 0");
  if ((q_norm_w == nullptr) != (k_norm_w == nullptr))
    return fail(DEC_ERR_INVALID_ARG, "q_norm_w and k_norm_w must both be set or both be null");
  if (B == 0) return ok();
  if (!q_in || !q_out || !k_new || !v_new || !k_cache || !v_cache || !pos)
    return fail(DEC_ERR_INVALID_ARG, "q, k_new, v_new, caches and pos must be non-null");
  if (!aligned16(q_in) || !aligned16(q_out) || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned16(k_cache) || !aligned16(v_cache) ||
      (q_norm_w && (!aligned16(q_norm_w) || !aligned16(k_norm_w))))
    return fail(DEC_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (k_cache == v_cache) return fail(DEC_ERR_INVALID_ARG, "k_cache and v_cache must differ");
  const size_t q_bytes = (size_t)B * Hq * D * 2;
  const char *qi = static_cast<const char *>(q_in);
  const char *qo = static_cast<const char *>(q_out);
  if (qi != qo && qi < qo + q_bytes && qo < qi + q_bytes)
    return fail(DEC_ERR_INVALID_ARG, "q_in and q_out must be the same buffer or not overlap");
  st = where_all({{q_in, "q_in", true}, {q_out, "q_out", true}, {k_new, "k_new", true},
                             {v_new, "v_new", true}, {q_norm_w, "q_norm_w", true},
                             {k_norm_w, "k_norm_w", true}, {k_cache, "k_cache", false},
                             {v_cache, "v_cache", false}, {pos, "pos", true},
                             {error_word, "error_word", true}});
  if (st != DEC_OK) return st;
  cudaError_t e = launch_qknorm_rope_append_strided(
      q_in, q_out, (size_t)Hq * D, k_new, v_new, (size_t)Hkv * D, q_norm_w, k_norm_w, k_cache,
      v_cache, pos, B, Hq, Hkv, D, T_cap, inv, layout == DEC_ROPE_INTERLEAVED, eps, error_word,
      as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qknorm_rope_kv_append launch");
  return ok();
}
}  // namespace

extern "C" {

dec_status dec_qknorm_rope_kv_append(void *q, const void *k_new, const void *v_new,
                                     const void *q_norm_w, const void *k_norm_w, void *k_cache,
                                     void *v_cache, const int32_t *pos, int B, int Hq, int Hkv,
                                     int D, int T_cap, float rope_theta, dec_rope_layout layout,
                                     const double *inv_freq, float eps, uint32_t *error_word,
                                     dec_stream_t stream) {
  return qknorm_rope_impl(q, q, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, pos, B, Hq,
                          Hkv, D, T_cap, rope_theta, layout, inv_freq, eps, error_word, stream);
}

dec_status dec_qknorm_rope_kv_append_out(const void *q_in, void *q_out, const void *k_new,
                                         const void *v_new, const void *q_norm_w,
                                         const void *k_norm_w, void *k_cache, void *v_cache,
                                         const int32_t *pos, int B, int Hq, int Hkv, int D,
                                         int T_cap, float rope_theta, dec_rope_layout layout,
                                         const double *inv_freq, float eps, uint32_t *error_word,
                                         dec_stream_t stream) {
  return qknorm_rope_impl(q_in, q_out, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, pos, B,
                          Hq, Hkv, D, T_cap, rope_theta, layout, inv_freq, eps, error_word,
                          stream);
}

dec_status dec_rope_inv_freq(int D, float rope_theta, dec_rope_scaling scaling, float factor,
                             double *inv_freq) {
  if (D != 64 && D != 128) return fail(DEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (inv_freq == nullptr) return fail(DEC_ERR_INVALID_ARG, "inv_freq must be non-null");
  if (!(rope_theta > 0.f) || std::isinf(rope_theta))
    return fail(DEC_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
  if (scaling != DEC_ROPE_SCALE_NONE && !(factor >= 1.f && std::isfinite(factor)))
    return fail(DEC_ERR_INVALID_ARG, "factor must be finite and >= 1");
  double base = (double)rope_theta, div = 1.0;
  switch (scaling) {
    case DEC_ROPE_SCALE_NONE:
      break;
    case DEC_ROPE_SCALE_LINEAR:  // positions divided by the factor
      div = (double)factor;
      break;
    case DEC_ROPE_SCALE_NTK:  // base enlarged so the slowest pair slows by the factor
      base *= std::pow((double)factor, (double)D / (double)(D - 2));
      break;
    default:
      return fail(DEC_ERR_INVALID_ARG, "unknown rope scaling %d", (int)scaling);
  }
  const InvFreq t = make_inv_freq(D, base);
  for (int i = 0; i < D / 2; ++i) inv_freq[i] = t.v[i] / div;
  return ok();
}

dec_status dec_rope_yarn_inv_freq(int D, float rope_theta, float factor, int original_context,
                                  float alpha, float beta, double *inv_freq,
                                  float *scale_mult) {
  if (D != 64 && D != 128) return fail(DEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (inv_freq == nullptr) return fail(DEC_ERR_INVALID_ARG, "inv_freq must be non-null");
  if (!(rope_theta > 0.f) || std::isinf(rope_theta))
    return fail(DEC_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
  if (!(factor >= 1.f && std::isfinite(factor)))
    return fail(DEC_ERR_INVALID_ARG, "factor must be finite and >= 1");
  if (original_context < 1)
    return fail(DEC_ERR_INVALID_ARG, "original_context = %d must be positive", original_context);
  if (!(alpha >= 0.f && beta > alpha && std::isfinite(beta)))
    return fail(DEC_ERR_INVALID_ARG, "need 0 <= alpha < beta, both finite");
  const InvFreq plain = make_inv_freq(D, (double)rope_theta);
  const double s = (double)factor, a = (double)alpha, b = (double)beta;
  for (int i = 0; i < D / 2; ++i) {
    const double f = plain.v[i];
    // turns of pair i over the original context, then the share of f it keeps
    const double turns = (double)original_context * f / 6.283185307179586;
    double keep = (turns - a) / (b - a);
    keep = keep < 0.0 ? 0.0 : (keep > 1.0 ? 1.0 : keep);
    inv_freq[i] = (1.0 - keep) * (f / s) + keep * f;
  }
  if (scale_mult != nullptr) {  // q and k each scaled by m: the logits by m^2
    const double m = s > 1.0 ? 0.1 * std::log(s) + 1.0 : 1.0;
    *scale_mult = (float)(m * m);
  }
  return ok();
}

dec_status dec_rope_yarn_softmax_scale(int D, float factor, float *scale) {
  if (D != 64 && D != 128) return fail(DEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (scale == nullptr) return fail(DEC_ERR_INVALID_ARG, "scale must be non-null");
  if (!(factor >= 1.f && std::isfinite(factor)))
    return fail(DEC_ERR_INVALID_ARG, "factor must be finite and >= 1");
  const double s = (double)factor;
  const double m = s > 1.0 ? 0.1 * std::log(s) + 1.0 : 1.0;
  *scale = (float)(m * m / std::sqrt((double)D));
  return ok();
}

int dec_decode_step_path(int B, int Hq, int Hkv, int D, int max_len, int window) {
  if (small_step_splits(B, Hq, Hkv, D, max_len, window) > 0) return DEC_STEP_SHORT;
  const int parts = dec_attn_default_parts(B, Hkv, D, max_len);
  return split_fused_fits(parts, current_device()) ? DEC_STEP_STREAM : DEC_STEP_THREE;
}

int dec_decode_step_launches(int B, int Hq, int Hkv, int D, int max_len, int window) {
  switch (dec_decode_step_path(B, Hq, Hkv, D, max_len, window)) {
    case DEC_STEP_SHORT: return 1;
    case DEC_STEP_STREAM: return 2;
    default: return 3;
  }
}

int dec_attn_default_parts(int B, int Hkv, int D, int max_len) {
  if (B <= 0 || Hkv <= 0 || (D != 64 && D != 128)) return 1;
  // one CTA per SM: the split kernel sizes its pipeline to fill an SM's shared memory
  const long long cap = (long long)sm_count(current_device());
  const long long rows = (long long)B * Hkv * (max_len < 0 ? 0 : max_len);
  long long need = (rows + kMinRowsPerPart - 1) / kMinRowsPerPart;
  if (need < 1) need = 1;
  return (int)(need < cap ? need : cap);
}

size_t dec_attn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len, int num_parts) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return 0;
  return workspace_bytes(B, Hq, Hkv, D, resolve_parts(num_parts, B, Hkv, D, max_len));
}

int dec_pick_num_splits(int B, int Hkv, int max_len, int sm_count) {
  if (B <= 0 || Hkv <= 0 || max_len <= 0) return 1;
  const long long cap = sm_count > 0 ? sm_count : sm_count_of_current();
  const long long rows = (long long)B * Hkv * max_len;
  long long need = (rows + kMinRowsPerPart - 1) / kMinRowsPerPart;
  if (need < 1) need = 1;
  return (int)(need < cap ? need : cap);
}

size_t dec_decode_workspace_bytes(int B, int Hq, int D, int max_splits) {
  if (B < 0 || Hq <= 0 || (D != 64 && D != 128)) return 0;
  const int P = max_splits > 0 ? max_splits : sm_count_of_current();
  // the workspace grows with the group size at a fixed Hq: take the largest supported
  size_t most = 0;
  for (int Hkv = 1; Hkv <= Hq; ++Hkv) {
    if (Hq % Hkv != 0 || Hq / Hkv > kSplitMaxG) continue;
    const size_t b = workspace_bytes(B, Hq, Hkv, D, P);
    if (b > most) most = b;
  }
  return most;
}

namespace {
// The split pass; with out_direct, pairs that lie in one piece are written to it.
dec_status split_impl(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *lens, int B, int Hq, int Hkv, int D, int T_cap, int max_len,
                      float scale, int num_parts, void *workspace, size_t ws_bytes,
                      void *out_direct, int window, dec_stream_t stream, bool dry = false,
                      bool fused = false) {
  dec_status st = check_attn_shape(B, Hq, Hkv, D, T_cap, max_len);
  if (st != DEC_OK) return st;
  if (num_parts < 0) return fail(DEC_ERR_INVALID_ARG, "num_parts = %d < 0", num_parts);
  if (B == 0) return ok();
  if (!q || !k_cache || !v_cache || !lens)
    return fail(DEC_ERR_INVALID_ARG, "q, caches and lens must be non-null");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(DEC_ERR_INVALID_ARG, "q and caches must be 16-byte aligned");
  if (!(std::isfinite(scale))) return fail(DEC_ERR_INVALID_ARG, "scale must be finite");
  const int parts = resolve_parts(num_parts, B, Hkv, D, max_len);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DEC_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  const size_t need = workspace_bytes(B, Hq, Hkv, D, parts);
  if (ws_bytes < need)
    return fail(DEC_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
  if (split_stages(D, Hq / Hkv, B, current_device()) < 2)
    return fail(DEC_ERR_UNSUPPORTED, "not enough shared memory for B = %d", B);
  if ((st = where_all({{q, "q", false}, {k_cache, "k_cache", false}, {v_cache, "v_cache", false},
                       {workspace, "workspace", false}, {lens, "lens", true},
                       {out_direct, "out", true}})) != DEC_OK)
    return st;
  CUtensorMap kmap, vmap, kmap8, vmap8;
  if ((st = encode_cache_map(&kmap, k_cache, B, Hkv, D, T_cap, kSplitBoxRows)) != DEC_OK) return st;
  if ((st = encode_cache_map(&vmap, v_cache, B, Hkv, D, T_cap, kSplitBoxRows)) != DEC_OK) return st;
  if ((st = encode_cache_map(&kmap8, k_cache, B, Hkv, D, T_cap, 8)) != DEC_OK) return st;
  if ((st = encode_cache_map(&vmap8, v_cache, B, Hkv, D, T_cap, 8)) != DEC_OK) return st;
  if (dry) return ok();  // every check passed; launch nothing
  const float s = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  const float scale_log2 = (float)((double)s * 1.4426950408889634);
  // the merge sizes its warp groups from the longest pair it can meet
  const int eff_len = (window > 0 && window < max_len) ? window : max_len;
  cudaError_t e = launch_gqa_split(kmap, vmap, kmap8, vmap8, q, lens, B, Hq, Hkv, D, T_cap,
                                   scale_log2, parts, workspace, out_direct, window,
                                   as_stream(stream), fused, eff_len);
  if (e != cudaSuccess) return cuda_fail(e, "gqa_decode_split launch");
  return ok();
}
}  // namespace

extern "C" dec_status dec_gqa_decode_split(const void *q, const void *k_cache,
                                           const void *v_cache, const int32_t *lens, int B,
                                           int Hq, int Hkv, int D, int T_cap, int max_len,
                                           float scale, int num_parts, void *workspace,
                                           size_t ws_bytes, dec_stream_t stream) {
  return split_impl(q, k_cache, v_cache, lens, B, Hq, Hkv, D, T_cap, max_len, scale, num_parts,
                    workspace, ws_bytes, nullptr, 0, stream);
}

dec_status dec_split_merge(const void *workspace, size_t ws_bytes, const int32_t *lens, void *out,
                           int B, int Hq, int Hkv, int D, int T_cap, int max_len, int num_parts,
                           dec_stream_t stream) {
  dec_status st = check_attn_shape(B, Hq, Hkv, D, T_cap, max_len);
  if (st != DEC_OK) return st;
  if (num_parts < 0) return fail(DEC_ERR_INVALID_ARG, "num_parts = %d < 0", num_parts);
  if (B == 0) return ok();
  if (!out || !lens) return fail(DEC_ERR_INVALID_ARG, "out and lens must be non-null");
  if (!aligned16(out)) return fail(DEC_ERR_INVALID_ARG, "out must be 16-byte aligned");
  const int parts = resolve_parts(num_parts, B, Hkv, D, max_len);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DEC_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  const size_t need = workspace_bytes(B, Hq, Hkv, D, parts);
  if (ws_bytes < need)
    return fail(DEC_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
  if ((st = where_all({{workspace, "workspace", false}, {out, "out", true}})) != DEC_OK) return st;
  cudaError_t e = launch_split_merge(workspace, out, B, Hq, Hkv, D, max_len, parts,
                                     as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "split_merge launch");
  return ok();
}

}  // extern "C"

namespace {
// The attention call for short contexts: the split and its merge in one launch (the
// one-launch step's kernel without its RMSNorm and rotation), with the split pass's
// argument rules.
dec_status attn_small_impl(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                           int T_cap, int max_len, float scale, int splits, void *workspace,
                           size_t ws_bytes, int window, dec_stream_t stream, bool dry) {
  if (!q || !k_cache || !v_cache || !lens)
    return fail(DEC_ERR_INVALID_ARG, "q, caches and lens must be non-null");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(DEC_ERR_INVALID_ARG, "q and caches must be 16-byte aligned");
  if (!(std::isfinite(scale))) return fail(DEC_ERR_INVALID_ARG, "scale must be finite");
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DEC_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  const size_t need = workspace_bytes(B, Hq, Hkv, D, resolve_parts(0, B, Hkv, D, max_len));
  if (ws_bytes < need)
    return fail(DEC_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
  dec_status st;
  if ((st = where_all({{q, "q", false}, {k_cache, "k_cache", false}, {v_cache, "v_cache", false},
                       {workspace, "workspace", false}, {lens, "lens", true},
                       {out, "out", true}})) != DEC_OK)
    return st;
  if (dry) return ok();
  const float s = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  cudaError_t e = launch_attn_small(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, splits,
                                    window, (float)((double)s * 1.4426950408889634),
                                    static_cast<uint32_t *>(workspace), as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "one-launch attention");
  return ok();
}

dec_status attn_impl(const void *q, const void *k_cache, const void *v_cache, const int32_t *lens,
                     void *out, int B, int Hq, int Hkv, int D, int T_cap, int max_len, float scale,
                     int num_parts, void *workspace, size_t ws_bytes, int window,
                     dec_stream_t stream, bool dry = false) {
  if (window < 0) return fail(DEC_ERR_INVALID_ARG, "window = %d < 0", window);
  if (B > 0 && !out) return fail(DEC_ERR_INVALID_ARG, "out must be non-null");
  if (B > 0 && !aligned16(out)) return fail(DEC_ERR_INVALID_ARG, "out must be 16-byte aligned");
  // short contexts with the split left to the library: one launch
  if (B > 0 && num_parts == 0) {
    dec_status st = check_attn_shape(B, Hq, Hkv, D, T_cap, max_len);
    if (st != DEC_OK) return st;
    const int small = small_step_splits(B, Hq, Hkv, D, max_len, window);
    if (small > 0)
      return attn_small_impl(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale,
                             small, workspace, ws_bytes, window, stream, dry);
  }
  const int parts = (B > 0 && num_parts >= 0) ? resolve_parts(num_parts, B, Hkv, D, max_len) : num_parts;
  // at most one CTA per SM: the split pass and its merge in one cooperative launch
  const bool fused = B > 0 && parts > 0 && split_fused_fits(parts, current_device());
  dec_status st = split_impl(q, k_cache, v_cache, lens, B, Hq, Hkv, D, T_cap, max_len, scale,
                             parts, workspace, ws_bytes, out, window, stream, dry, fused);
  if (st != DEC_OK || dry || fused) return st;
  // the merge sizes its warp groups from the longest pair it can meet
  const int eff_len = (window > 0 && window < max_len) ? window : max_len;
  return dec_split_merge(workspace, ws_bytes, lens, out, B, Hq, Hkv, D, T_cap, eff_len, parts,
                         stream);
}
}  // namespace

namespace decattn {
dec_status attn_check(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *lens, void *out, int B, int Hq, int Hkv, int D, int T_cap,
                      int max_len, float scale, int num_parts, void *workspace,
                      size_t ws_bytes) {
  return attn_impl(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale,
                   num_parts, workspace, ws_bytes, 0, nullptr, true);
}
dec_status check_reachable(const void *p, const char *name) { return where_ok(p, name, true); }
}  // namespace decattn

extern "C" {

dec_status dec_gqa_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *lens, void *out, int B, int Hq, int Hkv, int D,
                               int T_cap, int max_len, float scale, int num_parts, void *workspace,
                               size_t ws_bytes, dec_stream_t stream) {
  return attn_impl(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale,
                   num_parts, workspace, ws_bytes, 0, stream);
}

dec_status dec_gqa_decode_attn_window(const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *lens, void *out, int B, int Hq, int Hkv,
                                      int D, int T_cap, int max_len, int window, float scale,
                                      int num_parts, void *workspace, size_t ws_bytes,
                                      dec_stream_t stream) {
  if (window < 1) return fail(DEC_ERR_INVALID_ARG, "window = %d must be >= 1", window);
  return attn_impl(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale,
                   num_parts, workspace, ws_bytes, window, stream);
}

dec_status dec_decode_step(const void *x, void *residual, const void *norm_w, void *y, int hidden,
                           float eps, void *q, const void *k_new, const void *v_new,
                           const void *q_norm_w, const void *k_norm_w, void *k_cache,
                           void *v_cache, const int32_t *pos, const int32_t *lens, void *out,
                           int B, int Hq, int Hkv, int D, int T_cap, int max_len,
                           float rope_theta, dec_rope_layout layout, const double *inv_freq,
                           float scale, int window, int num_parts, void *workspace,
                           size_t ws_bytes, dec_stream_t stream) {
  // check everything before the first launch
  dec_status st = check_attn_shape(B, Hq, Hkv, D, T_cap, max_len);
  if (st != DEC_OK) return st;
  if (B == 0) return ok();
  if (hidden < 8 || hidden > 16384 || hidden % 8 != 0)
    return fail(DEC_ERR_UNSUPPORTED, "hidden = %d (need a multiple of 8 in [8, 16384])", hidden);
  const int parts = resolve_parts(num_parts < 0 ? 0 : num_parts, B, Hkv, D, max_len);
  if (num_parts < 0) return fail(DEC_ERR_INVALID_ARG, "num_parts = %d < 0", num_parts);
  if (window < 0) return fail(DEC_ERR_INVALID_ARG, "window = %d < 0", window);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DEC_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  if (ws_bytes < workspace_bytes(B, Hq, Hkv, D, parts))
    return fail(DEC_ERR_WORKSPACE, "workspace too small");
  // K1 and K2 share one launch; their arguments are checked by the standalone calls'
  // rules first
  if (!x || !norm_w || !y || !q || !k_new || !v_new || !k_cache || !v_cache || !pos)
    return fail(DEC_ERR_INVALID_ARG, "x, norm_w, y, q, k_new, v_new, caches and pos must be non-null");
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(y) || (residual && !aligned16(residual)) ||
      !aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || (q_norm_w && !aligned16(q_norm_w)) || (k_norm_w && !aligned16(k_norm_w)))
    return fail(DEC_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (y == x || (residual != nullptr && y == residual))
    return fail(DEC_ERR_INVALID_ARG, "y may not alias x or residual");
  if (k_cache == v_cache) return fail(DEC_ERR_INVALID_ARG, "k_cache and v_cache must differ");
  if ((q_norm_w == nullptr) != (k_norm_w == nullptr))
    return fail(DEC_ERR_INVALID_ARG, "q_norm_w and k_norm_w must both be set or both be null");
  if (!(eps >= 0.f)) return fail(DEC_ERR_INVALID_ARG, "eps must be >= 0");
  InvFreq inv;
  if ((st = rope_table(D, rope_theta, inv_freq, &inv)) != DEC_OK) return st;
  if (layout != DEC_ROPE_NEOX && layout != DEC_ROPE_INTERLEAVED)
    return fail(DEC_ERR_INVALID_ARG, "unknown rope layout %d", (int)layout);
  if (!(std::isfinite(scale))) return fail(DEC_ERR_INVALID_ARG, "scale must be finite");
  // short contexts run as one launch, which reads and writes q with plain loads and
  // stores; otherwise the split pass reads q with bulk copies
  const int small = small_step_splits(B, Hq, Hkv, D, max_len, window);
  if ((st = where_all({{x, "x", true}, {residual, "residual", true}, {norm_w, "norm_w", true},
                       {y, "y", true}, {q, "q", small > 0}, {k_new, "k_new", true},
                       {v_new, "v_new", true}, {q_norm_w, "q_norm_w", true},
                       {k_norm_w, "k_norm_w", true}, {pos, "pos", true},
                       {k_cache, "k_cache", false}, {v_cache, "v_cache", false},
                       {workspace, "workspace", false}})) != DEC_OK)
    return st;
  // short contexts: the whole step in one launch
  if (small > 0) {
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
    cudaError_t e = launch_decode_small(
        x, residual, norm_w, y, hidden, eps, q, k_new, v_new, q_norm_w, k_norm_w, k_cache,
        v_cache, pos, lens, out, B, Hq, Hkv, D, T_cap, small, window,
        (float)((double)sc * 1.4426950408889634), inv, layout == DEC_ROPE_INTERLEAVED, static_cast<uint32_t *>(workspace), as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "one-launch decode step");
    return ok();
  }
  cudaError_t e = launch_rms_rope_fused(x, residual, norm_w, y, hidden, eps, q, k_new, v_new,
                                        q_norm_w, k_norm_w, k_cache, v_cache, pos, B, Hq, Hkv, D,
                                        T_cap, inv, layout == DEC_ROPE_INTERLEAVED,
                                        static_cast<uint32_t *>(workspace), as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm + rope launch");
  return attn_impl(q, k_cache, v_cache, lens, out, B, Hq, Hkv, D, T_cap, max_len, scale, parts,
                   workspace, ws_bytes, window, stream);
}

}  // extern "C"

// ------------------------------------------------------------ projections ---
namespace {

// A row-major [rows, inner] bf16 matrix as a 2-D tensor, boxes of 64 x box_rows,
// 128-byte swizzle; rows past the end read as zeros.
dec_status encode_matrix_map(CUtensorMap *map, const void *base, int rows, int inner,
                             int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return fail(DEC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DEC_OK;
}

bool overlaps(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + b_bytes && pb < pa + a_bytes;
}

dec_status check_linear_shape(int B, int N, int K) {
  if (B < 0) return fail(DEC_ERR_INVALID_ARG, "B = %d < 0", B);
  if (N < 128 || N % 128 != 0)
    return fail(DEC_ERR_UNSUPPORTED, "N = %d (need a positive multiple of 128)", N);
  if (K < 64 || K % 64 != 0)
    return fail(DEC_ERR_UNSUPPORTED, "K = %d (need a positive multiple of 64)", K);
  if ((long long)B * N >= (1ll << 31) || (long long)B * K >= (1ll << 31) ||
      (long long)N * K >= (1ll << 40))
    return fail(DEC_ERR_UNSUPPORTED, "projection too large");
  return DEC_OK;
}

int check_k_split(int k_split, int K) {
  return k_split < 0 || k_split > 8 || (k_split > 0 && k_split > K / 64);
}

// y = x w^T (+ residual).
dec_status linear_impl(const void *x, const void *w, const void *residual, void *y, int B, int N,
                       int K, int k_split, uint32_t *error_word, dec_stream_t stream) {
  dec_status st = check_linear_shape(B, N, K);
  if (st != DEC_OK) return st;
  if (check_k_split(k_split, K))
    return fail(DEC_ERR_INVALID_ARG, "k_split = %d (0 = automatic, else 1 .. min(8, K / 64))",
                k_split);
  if (B == 0) return ok();
  if (!x || !w || !y) return fail(DEC_ERR_INVALID_ARG, "x, w and y must be non-null");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)))
    return fail(DEC_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const size_t y_bytes = (size_t)B * N * 2;
  if (overlaps(y, y_bytes, x, (size_t)B * K * 2) || overlaps(y, y_bytes, w, (size_t)N * K * 2))
    return fail(DEC_ERR_INVALID_ARG, "y may not overlap x or w");
  if (residual != nullptr && residual != y && overlaps(y, y_bytes, residual, y_bytes))
    return fail(DEC_ERR_INVALID_ARG, "residual must be y itself or not overlap it");
  if ((st = where_all({{x, "x", false}, {w, "w", false}, {residual, "residual", true},
                       {y, "y", true}, {error_word, "error_word", true}})) != DEC_OK)
    return st;
  const LinPlan plan = linear_plan(B, N, K, current_device(), false, k_split);
  CUtensorMap wmap, xmap;
  if ((st = encode_matrix_map(&wmap, w, N, K, 128)) != DEC_OK) return st;
  if ((st = encode_matrix_map(&xmap, x, B, K, plan.nb)) != DEC_OK) return st;
  cudaError_t e = launch_linear(wmap, xmap, residual, y, B, N, K, plan, error_word,
                                as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "linear launch");
  return ok();
}

// The RMSNorm prologue's inputs: x and the optional residual r [B, K], the norm weight
// [K], the optional h_out [B, K] for x + r. Checked against each other and against the
// projection's output `out` (out_bytes), then given their tensor maps.
struct NormIn {
  const void *x, *residual, *norm_w;
  void *h_out;
  float eps;
};

dec_status check_norm_in(const NormIn &n, int B, int K, int nb, const void *out,
                         size_t out_bytes, CUtensorMap *xmap, CUtensorMap *rmap, LinNorm *ln) {
  if (!(n.eps >= 0.f)) return fail(DEC_ERR_INVALID_ARG, "eps must be >= 0");
  if (!n.x || !n.norm_w) return fail(DEC_ERR_INVALID_ARG, "x and norm_w must be non-null");
  if (!aligned16(n.x) || !aligned16(n.norm_w) || (n.residual && !aligned16(n.residual)) ||
      (n.h_out && !aligned16(n.h_out)))
    return fail(DEC_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const size_t act = (size_t)B * K * 2;
  if (overlaps(out, out_bytes, n.x, act) || (n.residual && overlaps(out, out_bytes, n.residual, act)))
    return fail(DEC_ERR_INVALID_ARG, "the projection's output may not overlap x or residual");
  if (n.h_out && (overlaps(n.h_out, act, n.x, act) ||
                  (n.residual && overlaps(n.h_out, act, n.residual, act)) ||
                  overlaps(n.h_out, act, out, out_bytes)))
    return fail(DEC_ERR_INVALID_ARG,
                "h_out may not overlap x, residual or the projection's output (the other "
                "CTAs still read them)");
  dec_status st = where_all({{n.x, "x", false}, {n.residual, "residual", false},
                             {n.norm_w, "norm_w", false}, {n.h_out, "h_out", true}});
  if (st != DEC_OK) return st;
  if ((st = encode_matrix_map(xmap, n.x, B, K, nb)) != DEC_OK) return st;
  *rmap = *xmap;
  if (n.residual && (st = encode_matrix_map(rmap, n.residual, B, K, nb)) != DEC_OK) return st;
  ln->norm_w = n.norm_w;
  ln->h_out = n.h_out;
  ln->inv_k = 1.0f / (float)K;
  ln->eps = n.eps;
  ln->has_r = n.residual != nullptr;
  return DEC_OK;
}

// y = RMSNorm(x + residual) w^T, the normalisation formed inside the projection.
dec_status norm_linear_impl(const NormIn &n, const void *w, void *y, int B, int N, int K,
                            int k_split, uint32_t *error_word, dec_stream_t stream) {
  dec_status st = check_linear_shape(B, N, K);
  if (st != DEC_OK) return st;
  if (check_k_split(k_split, K))
    return fail(DEC_ERR_INVALID_ARG, "k_split = %d (0 = automatic, else 1 .. min(8, K / 64))",
                k_split);
  if (B == 0) return ok();
  if (!w || !y) return fail(DEC_ERR_INVALID_ARG, "w and y must be non-null");
  if (!aligned16(w) || !aligned16(y))
    return fail(DEC_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const size_t y_bytes = (size_t)B * N * 2;
  if (overlaps(y, y_bytes, w, (size_t)N * K * 2))
    return fail(DEC_ERR_INVALID_ARG, "y may not overlap w");
  const LinPlan plan = linear_plan(B, N, K, current_device(), true, k_split);
  CUtensorMap wmap, xmap, rmap;
  LinNorm ln{};
  if ((st = check_norm_in(n, B, K, plan.nb, y, y_bytes, &xmap, &rmap, &ln)) != DEC_OK) return st;
  if ((st = where_all({{w, "w", false}, {y, "y", true}, {error_word, "error_word", true}})) !=
      DEC_OK)
    return st;
  if ((st = encode_matrix_map(&wmap, w, N, K, 128)) != DEC_OK) return st;
  cudaError_t e = launch_linear_norm(wmap, xmap, rmap, ln, y, B, N, K, plan, error_word,
                                     as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "linear launch");
  return ok();
}

// The packed QKV projection with the rotation as its epilogue (head_dim 128), of y, or
// (norm != nullptr) of RMSNorm(x + residual) formed in its prologue, y unused.
dec_status qkv_rot_impl(const void *y, const void *w_qkv, const void *q_norm_w,
                        const void *k_norm_w, void *q_out, void *k_cache, void *v_cache,
                        const int32_t *pos, int B, int hidden, int Hq, int Hkv, int D, int T_cap,
                        float rope_theta, dec_rope_layout layout, const double *inv_freq,
                        float eps, uint32_t *error_word, dec_stream_t stream,
                        const NormIn *norm = nullptr) {
  const int nqkv = (Hq + 2 * Hkv) * D;
  dec_status st = check_linear_shape(B, nqkv, hidden);
  if (st != DEC_OK) return st;
  if (D != 128) return fail(DEC_ERR_UNSUPPORTED, "the fused rotation needs head_dim 128");
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(DEC_ERR_INVALID_ARG, "need Hq, Hkv > 0 and Hq %% Hkv == 0");
  if (T_cap <= 0) return fail(DEC_ERR_INVALID_ARG, "T_cap = %d must be positive", T_cap);
  InvFreq inv;
  if ((st = rope_table(D, rope_theta, inv_freq, &inv)) != DEC_OK) return st;
  if (layout != DEC_ROPE_NEOX && layout != DEC_ROPE_INTERLEAVED)
    return fail(DEC_ERR_INVALID_ARG, "unknown rope layout %d", (int)layout);
  if (!(eps >= 0.f)) return fail(DEC_ERR_INVALID_ARG, "eps must be >= 0");
  if ((q_norm_w == nullptr) != (k_norm_w == nullptr))
    return fail(DEC_ERR_INVALID_ARG, "q_norm_w and k_norm_w must both be set or both be null");
  if (B == 0) return ok();
  if (norm != nullptr) y = norm->x;
  if (!y || !w_qkv || !q_out || !k_cache || !v_cache || !pos)
    return fail(DEC_ERR_INVALID_ARG, "y, w_qkv, q_out, caches and pos must be non-null");
  if (!aligned16(y) || !aligned16(w_qkv) || !aligned16(q_out) || !aligned16(k_cache) ||
      !aligned16(v_cache) || (q_norm_w && (!aligned16(q_norm_w) || !aligned16(k_norm_w))))
    return fail(DEC_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (k_cache == v_cache) return fail(DEC_ERR_INVALID_ARG, "k_cache and v_cache must differ");
  const LinPlan plan = linear_plan(B, nqkv, hidden, current_device(), norm != nullptr);
  CUtensorMap xmap, rmap;
  LinNorm ln{};
  if (norm != nullptr) {
    const size_t q_bytes = (size_t)B * Hq * D * 2;
    if ((st = check_norm_in(*norm, B, hidden, plan.nb, q_out, q_bytes, &xmap, &rmap, &ln)) !=
        DEC_OK)
      return st;
    const size_t act = (size_t)B * hidden * 2;
    if (norm->h_out && overlaps(norm->h_out, act, q_out, q_bytes))
      return fail(DEC_ERR_INVALID_ARG, "h_out may not overlap q_out");
  }
  if ((st = where_all({{y, "y", false}, {w_qkv, "w_qkv", false}, {q_norm_w, "q_norm_w", true},
                       {k_norm_w, "k_norm_w", true}, {q_out, "q_out", true},
                       {k_cache, "k_cache", false}, {v_cache, "v_cache", false},
                       {pos, "pos", true}, {error_word, "error_word", true}})) != DEC_OK)
    return st;
  QkvRotArgs rot{};
  rot.q_out = q_out;
  rot.k_cache = k_cache;
  rot.v_cache = v_cache;
  rot.pos = pos;
  rot.q_norm_w = q_norm_w;
  rot.k_norm_w = k_norm_w;
  rot.Hq = Hq;
  rot.Hkv = Hkv;
  rot.T_cap = T_cap;
  rot.interleaved = layout == DEC_ROPE_INTERLEAVED;
  rot.eps = eps;
  const RopeTurns turns = make_rope_turns(D, inv);
  for (int i = 0; i < 64; ++i) rot.turns[i] = turns.v[i];
  CUtensorMap wmap;
  if ((st = encode_matrix_map(&wmap, w_qkv, nqkv, hidden, 128)) != DEC_OK) return st;
  if (norm == nullptr && (st = encode_matrix_map(&xmap, y, B, hidden, plan.nb)) != DEC_OK)
    return st;
  cudaError_t e = launch_linear_qkv_rot(wmap, xmap, B, nqkv, hidden, plan, rot, error_word,
                                        as_stream(stream), norm ? &rmap : nullptr,
                                        norm ? &ln : nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "qkv projection launch");
  return ok();
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Sublayer workspace: [attention workspace | y | qkv | q_rot | attn].
struct SublayerLayout {
  size_t y, qkv, q_rot, attn, total;
};

SublayerLayout sublayer_layout(int B, int hidden, int Hq, int Hkv, int D, int parts) {
  SublayerLayout L{};
  const int nqkv = (Hq + 2 * Hkv) * D;
  L.y = align256(workspace_bytes(B, Hq, Hkv, D, parts));
  L.qkv = L.y + align256((size_t)B * hidden * 2);
  L.q_rot = L.qkv + align256((size_t)B * nqkv * 2);
  L.attn = L.q_rot + align256((size_t)B * Hq * D * 2);
  L.total = L.attn + align256((size_t)B * Hq * D * 2);
  return L;
}

}  // namespace

extern "C" {

dec_status dec_linear_plan(int B, int N, int K, int *batch_tile, int *k_split) {
  dec_status st = check_linear_shape(B, N, K);
  if (st != DEC_OK) return st;
  const LinPlan plan = B == 0 ? LinPlan{linear_batch_tile(0), 1}
                              : linear_plan(B, N, K, current_device());
  if (batch_tile) *batch_tile = plan.nb;
  if (k_split) *k_split = plan.splits;
  return ok();
}

dec_status dec_linear(const void *x, const void *w, const void *residual, void *y, int B, int N,
                      int K, int k_split, uint32_t *error_word, dec_stream_t stream) {
  return linear_impl(x, w, residual, y, B, N, K, k_split, error_word, stream);
}

dec_status dec_qkv_proj_rope_append(const void *y, const void *w_qkv, const void *q_norm_w,
                                    const void *k_norm_w, void *q_out, void *k_cache,
                                    void *v_cache, const int32_t *pos, int B, int hidden, int Hq,
                                    int Hkv, int D, int T_cap, float rope_theta,
                                    dec_rope_layout layout, const double *inv_freq, float eps,
                                    uint32_t *error_word, dec_stream_t stream) {
  return qkv_rot_impl(y, w_qkv, q_norm_w, k_norm_w, q_out, k_cache, v_cache, pos, B, hidden, Hq,
                      Hkv, D, T_cap, rope_theta, layout, inv_freq, eps, error_word, stream);
}

dec_status dec_norm_linear(const void *x, const void *residual, const void *norm_w, void *h_out,
                           const void *w, void *y, int B, int N, int K, float eps, int k_split,
                           uint32_t *error_word, dec_stream_t stream) {
  const NormIn n{x, residual, norm_w, h_out, eps};
  return norm_linear_impl(n, w, y, B, N, K, k_split, error_word, stream);
}

dec_status dec_norm_qkv_proj_rope_append(const void *x, const void *residual,
                                         const void *norm_w, void *h_out, const void *w_qkv,
                                         const void *q_norm_w, const void *k_norm_w, void *q_out,
                                         void *k_cache, void *v_cache, const int32_t *pos, int B,
                                         int hidden, int Hq, int Hkv, int D, int T_cap,
                                         float rope_theta, dec_rope_layout layout,
                                         const double *inv_freq, float eps,
                                         uint32_t *error_word, dec_stream_t stream) {
  const NormIn n{x, residual, norm_w, h_out, eps};
  return qkv_rot_impl(x, w_qkv, q_norm_w, k_norm_w, q_out, k_cache, v_cache, pos, B, hidden, Hq,
                      Hkv, D, T_cap, rope_theta, layout, inv_freq, eps, error_word, stream, &n);
}

size_t dec_attn_sublayer_workspace_bytes(int B, int hidden, int Hq, int Hkv, int D, int max_len,
                                         int num_parts) {
  if (B < 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (D != 64 && D != 128))
    return 0;
  return sublayer_layout(B, hidden, Hq, Hkv, D, resolve_parts(num_parts, B, Hkv, D, max_len))
      .total;
}

dec_status dec_attn_sublayer_layout(int B, int hidden, int Hq, int Hkv, int D, int max_len,
                                    int num_parts, size_t *offsets) {
  if (offsets == nullptr) return fail(DEC_ERR_INVALID_ARG, "offsets must be non-null");
  if (B < 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (D != 64 && D != 128) ||
      num_parts < 0)
    return fail(DEC_ERR_INVALID_ARG, "bad shape");
  const SublayerLayout L =
      sublayer_layout(B, hidden, Hq, Hkv, D, resolve_parts(num_parts, B, Hkv, D, max_len));
  offsets[0] = L.y;
  offsets[1] = L.qkv;
  offsets[2] = L.q_rot;
  offsets[3] = L.attn;
  offsets[4] = L.total;
  return ok();
}

dec_status dec_attn_sublayer(const void *x, void *residual, const void *norm_w, int hidden,
                             float eps, const void *w_qkv, const void *w_o, const void *q_norm_w,
                             const void *k_norm_w, void *k_cache, void *v_cache,
                             const int32_t *pos, const int32_t *lens, void *out, int B, int Hq,
                             int Hkv, int D, int T_cap, int max_len, float rope_theta,
                             dec_rope_layout layout, const double *inv_freq, float scale,
                             int window, int num_parts, void *workspace, size_t ws_bytes,
                             dec_stream_t stream) {
  dec_status st = check_attn_shape(B, Hq, Hkv, D, T_cap, max_len);
  if (st != DEC_OK) return st;
  const int nqkv = (Hq + 2 * Hkv) * D;
  if (hidden < 128 || hidden % 128 != 0 || hidden > 16384)
    return fail(DEC_ERR_UNSUPPORTED, "hidden = %d (need a multiple of 128 in [128, 16384])",
                hidden);
  if (nqkv % 128 != 0)
    return fail(DEC_ERR_UNSUPPORTED, "(Hq + 2 Hkv) * D = %d is not a multiple of 128", nqkv);
  if (num_parts < 0) return fail(DEC_ERR_INVALID_ARG, "num_parts = %d < 0", num_parts);
  if (window < 0) return fail(DEC_ERR_INVALID_ARG, "window = %d < 0", window);
  if (!(eps >= 0.f)) return fail(DEC_ERR_INVALID_ARG, "eps must be >= 0");
  InvFreq inv;
  if ((st = rope_table(D, rope_theta, inv_freq, &inv)) != DEC_OK) return st;
  if (layout != DEC_ROPE_NEOX && layout != DEC_ROPE_INTERLEAVED)
    return fail(DEC_ERR_INVALID_ARG, "unknown rope layout %d", (int)layout);
  if ((q_norm_w == nullptr) != (k_norm_w == nullptr))
    return fail(DEC_ERR_INVALID_ARG, "q_norm_w and k_norm_w must both be set or both be null");
  if (!(std::isfinite(scale))) return fail(DEC_ERR_INVALID_ARG, "scale must be finite");
  if (B == 0) return ok();
  if (!x || !norm_w || !w_qkv || !w_o || !k_cache || !v_cache || !pos || !lens || !out)
    return fail(DEC_ERR_INVALID_ARG,
                "x, norm_w, w_qkv, w_o, caches, pos, lens and out must be non-null");
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(w_qkv) || !aligned16(w_o) ||
      !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (residual && !aligned16(residual)) || (q_norm_w && !aligned16(q_norm_w)) ||
      (k_norm_w && !aligned16(k_norm_w)))
    return fail(DEC_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (k_cache == v_cache) return fail(DEC_ERR_INVALID_ARG, "k_cache and v_cache must differ");
  const size_t act = (size_t)B * hidden * 2;
  if (overlaps(out, act, x, act) || (residual && overlaps(out, act, residual, act)))
    return fail(DEC_ERR_INVALID_ARG, "out may not overlap x or residual");
  const int parts = resolve_parts(num_parts, B, Hkv, D, max_len);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DEC_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  const SublayerLayout L = sublayer_layout(B, hidden, Hq, Hkv, D, parts);
  if (ws_bytes < L.total)
    return fail(DEC_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, L.total);
  if (split_stages(D, Hq / Hkv, B, current_device()) < 2)
    return fail(DEC_ERR_UNSUPPORTED, "not enough shared memory for B = %d", B);
  // RMSNorm reads x and the residual and the output projection's epilogue reads the
  // residual and writes out with plain loads and stores; the weights and the caches
  // are read with bulk copies
  if ((st = where_all({{x, "x", true}, {residual, "residual", true}, {norm_w, "norm_w", true},
                       {out, "out", true}, {pos, "pos", true}, {lens, "lens", true},
                       {w_qkv, "w_qkv", false}, {w_o, "w_o", false},
                       {k_cache, "k_cache", false}, {v_cache, "v_cache", false},
                       {workspace, "workspace", false}})) != DEC_OK)
    return st;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint32_t *err = reinterpret_cast<uint32_t *>(ws);
  void *y = ws + L.y, *qkv = ws + L.qkv, *q_rot = ws + L.q_rot, *attn = ws + L.attn;
  cudaStream_t s = as_stream(stream);

  // h = x + residual (kept in `residual`), y = RMSNorm(h). A launch of its own: the
  // projections' RMSNorm prologue (dec_norm_*) measured no faster at decode batches and
  // slower at large ones, where every feature tile re-forms the same operand.
  cudaError_t e = launch_rmsnorm_residual(x, residual, norm_w, y, B, hidden, eps, s);
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm_residual launch");
  if (D == 128) {
    // [q | k | v] = y Wqkv^T with QK-norm + RoPE + the K/V append as its epilogue
    if ((st = qkv_rot_impl(y, w_qkv, q_norm_w, k_norm_w, q_rot, k_cache, v_cache, pos, B, hidden,
                           Hq, Hkv, D, T_cap, rope_theta, layout, inv_freq, eps, err,
                           stream)) != DEC_OK)
      return st;
  } else {
    // packed [q | k | v] = y Wqkv^T, then the rotation reading its column blocks
    if ((st = linear_impl(y, w_qkv, nullptr, qkv, B, nqkv, hidden, 0, err, stream)) != DEC_OK)
      return st;
    const size_t row = (size_t)nqkv;
    e = launch_qknorm_rope_append_strided(
        qkv, q_rot, row, static_cast<uint8_t *>(qkv) + (size_t)Hq * D * 2,
        static_cast<uint8_t *>(qkv) + (size_t)(Hq + Hkv) * D * 2, row, q_norm_w, k_norm_w,
        k_cache, v_cache, pos, B, Hq, Hkv, D, T_cap, inv, layout == DEC_ROPE_INTERLEAVED, eps,
        err, s);
    if (e != cudaSuccess) return cuda_fail(e, "qknorm_rope_kv_append launch");
  }
  // attention over the cache
  // (num_parts = 0: one launch for short contexts, else the split count `parts` resolves to)
  if ((st = attn_impl(q_rot, k_cache, v_cache, lens, attn, B, Hq, Hkv, D, T_cap, max_len, scale,
                      num_parts, workspace, L.y, window, stream)) != DEC_OK)
    return st;
  // out = h + attn Wo^T
  const void *h = residual != nullptr ? residual : x;
  return linear_impl(attn, w_o, h, out, B, hidden, Hq * D, 0, err, stream);
}

}  // extern "C"

// ------------------------------------------------------------------ sampler ---
extern "C" dec_status dec_sample(const float *logits, const int32_t *sampled_ids, int L,
                                 const float *u, int32_t *tokens, int B, int V, float penalty,
                                 float temperature, float top_p, int top_k, dec_stream_t stream) {
  if (B < 0) return fail(DEC_ERR_INVALID_ARG, "B = %d < 0", B);
  if (B > 65535) return fail(DEC_ERR_UNSUPPORTED, "B = %d rows > 65535 per call", B);
  if (V < 1) return fail(DEC_ERR_INVALID_ARG, "V = %d < 1", V);
  if (!sampler_supports(V))
    return fail(DEC_ERR_UNSUPPORTED, "V = %d is too large for the sampler", V);
  if (L < 0) return fail(DEC_ERR_INVALID_ARG, "L = %d < 0", L);
  if (!(penalty > 0.f) || std::isinf(penalty))
    return fail(DEC_ERR_INVALID_ARG, "penalty must be finite and > 0");
  if (std::isnan(temperature) || std::isinf(temperature))
    return fail(DEC_ERR_INVALID_ARG, "temperature must be finite");
  if (!(top_p > 0.f && top_p <= 1.f))
    return fail(DEC_ERR_INVALID_ARG, "top_p must lie in (0, 1]");
  if (top_k < 0) return fail(DEC_ERR_INVALID_ARG, "top_k = %d < 0", top_k);
  if (B == 0) return ok();
  if (!logits || !tokens) return fail(DEC_ERR_INVALID_ARG, "logits and tokens must be non-null");
  if (L > 0 && !sampled_ids)
    return fail(DEC_ERR_INVALID_ARG, "sampled_ids must be non-null when L > 0");
  if (temperature > 0.f && !u)
    return fail(DEC_ERR_INVALID_ARG, "u must be non-null when temperature > 0");
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(tokens) & 3u) ||
      (sampled_ids && (reinterpret_cast<uintptr_t>(sampled_ids) & 3u)) ||
      (u && (reinterpret_cast<uintptr_t>(u) & 3u)))
    return fail(DEC_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  if ((long long)B * V >= (1ll << 40)) return fail(DEC_ERR_UNSUPPORTED, "B * V too large");
  const dec_status st = where_all({{logits, "logits", true}, {tokens, "tokens", true},
                                   {L > 0 ? sampled_ids : nullptr, "sampled_ids", true},
                                   {temperature > 0.f ? u : nullptr, "u", true}});
  if (st != DEC_OK) return st;
  cudaError_t e = launch_sampler(logits, L > 0 ? sampled_ids : nullptr, L, u, tokens, B, V,
                                 penalty, temperature, top_p, top_k, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sampler launch");
  return ok();
}
