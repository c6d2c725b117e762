"""CPU oracle of the decode-step attention block (test infrastructure only).

Plain float64 numpy statements of what each step of the block computes. Nothing
here is blocked, fused or reordered beyond the definitions below, so each
function can be checked against the pages by eye. The oracle is independent of
the CUDA path: it shares no code, table or constant with it, and only the test
suite, the smoke check and the benchmark's CPU-baseline leg may import it.

Inputs are float64 arrays holding the exact values of the bf16 inputs; outputs
are float64 (the comparison with bf16 results happens in the tests).

Sources, by page and section:
* fusedtok 1.0.1 README, "Operators" table: RMSNorm (+residual) with a fused
  residual add; RoPE in interleaved and NeoX layouts with a kv-cache position
  offset; attention_decode = single-token causal attention with GQA over a
  contiguous kv-cache, online softmax, flash-decoding split over long caches,
  per-sequence lengths.
* fusedtok 1.0.1 README, "Usage": call shapes (q [B,Hq,D], caches [B,Hkv,T,D],
  lens [B] int32), ``rmsnorm(h, w, residual=h)``, ``rope(q, pos_offset=..., neox=True)``;
  "Benchmarks": the attention comparator expands heads with repeat_interleave,
  i.e. query head h reads KV head h // (Hq/Hkv); bf16 tensors are computed in
  float32 and converted at the load/store boundary.
* cutileGPT README, "Why tiles": the RMSNorm tile kernel,
  rstd = 1 / sqrt(sum(x*x)/N + eps), y = x * rstd * w; "The current runtime
  includes": fused QK-Norm + RoPE + KV-cache writes.

Readings taken where the pages are silent (each is listed in the design notes):
* RoPE: inv_freq_i = theta^(-2i/D) for i in [0, D/2); the pair (a, b) rotates to
  (a cos phi - b sin phi, a sin phi + b cos phi) with phi = pos * inv_freq_i; NeoX
  pairs element i with i + D/2, interleaved pairs 2i with 2i + 1; all D dims rotate.
* RoPE context extension (PyGPUkit 0.2.18 page, "Positional Encoding Operations",
  names only): linear interpolation divides every frequency by the factor s; the
  NTK-aware table is the plain one of the base theta * s^(D/(D-2)); YaRN blends the
  two per pair by how often it turns over the original context, and multiplies the
  rotated q and k by 0.1 ln(s) + 1.
* QK-norm: RMSNorm over head_dim with one [D] weight shared by all heads, applied
  before RoPE, same eps as the block.
* The new token sits at cache slot pos_b and is the last of len_b = pos_b + 1
  attended tokens; its RoPE position is pos_b.
* Attention scale 1/sqrt(D) unless given; a sequence of length 0 yields zeros.
* The fused residual add writes x + residual back as the new residual, and the
  norm is taken of the unrounded sum.
"""
from __future__ import annotations

import numpy as np

NEOX = "neox"
INTERLEAVED = "interleaved"


# ---------------------------------------------------------------- RMSNorm ---
def rms_norm(s: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: s / sqrt(mean(s^2) + eps) * w.

    cutileGPT README, "Why tiles" (rstd = 1/sqrt(sum(x*x)/N + eps); y = x*rstd*w).
    """
    s = np.asarray(s, dtype=np.float64)
    ms = np.mean(s * s, axis=-1, keepdims=True)
    return s / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rmsnorm_residual(x, residual, w, eps):
    """Fused residual add + RMSNorm.

    fusedtok README, "Operators" (RMSNorm (+residual): fused residual add) and
    "Usage" (``h = ft.rmsnorm(h, w, residual=h)``). Returns (y, new_residual) where
    new_residual = x + residual (or x when residual is None) and y is the RMSNorm of
    that sum.
    """
    x = np.asarray(x, dtype=np.float64)
    s = x if residual is None else x + np.asarray(residual, dtype=np.float64)
    return rms_norm(s, w, eps), s


# -------------------------------------------------------------------- RoPE ---
def rope_inv_freq(D: int, theta: float) -> np.ndarray:
    """inv_freq_i = theta^(-2i/D), i = 0 .. D/2-1 (fusedtok README, "Operators", RoPE)."""
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / D)


def yarn_ramp(r, alpha: float, beta: float):
    """The YaRN ramp gamma(r): 0 below alpha, 1 above beta, linear between (YaRN,
    Peng et al. 2023, "NTK-by-parts" interpolation; named on the PyGPUkit 0.2.18 page,
    "Positional Encoding Operations", as rope_init_yarn)."""
    r = np.asarray(r, dtype=np.float64)
    return np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)


def yarn_attention_factor(factor: float) -> float:
    """YaRN's attention temperature: the rotated q and k are both multiplied by
    sqrt(1/t) = 0.1 ln(s) + 1, so the logits by its square (published method; factor
    1 leaves them unchanged)."""
    return 0.1 * np.log(np.float64(factor)) + 1.0 if factor > 1.0 else 1.0


def rope_scaled_inv_freq(D: int, theta: float, scaling: str = "none",
                         factor: float = 1.0, original_context: int = 4096,
                         alpha: float = 1.0, beta: float = 32.0) -> np.ndarray:
    """Frequency tables for context extension.

    PyGPUkit 0.2.18 page, "Positional Encoding Operations" (rope_init_linear: linear
    position interpolation; rope_init_ntk_aware: NTK-aware RoPE for context
    extension). The page names the tables and gives no formula; the readings, from
    the usual statements of the two methods, with s = ``factor``:

    * "linear": every position is divided by s before the rotation, so pair i turns
      by (p / s) theta^(-2i/D): the plain table divided by s;
    * "ntk": the plain table of the larger base theta * s^(D / (D - 2)). The fastest
      pair (i = 0) keeps frequency 1 and the slowest (i = D/2 - 1) turns exactly s
      times slower; the pairs between are spread geometrically as before.
    * "yarn" (rope_init_yarn, "dimension-wise interpolation"; the published YaRN
      method): pair i of the plain table, frequency f_i and wavelength 2 pi / f_i,
      turns r_i = original_context * f_i / (2 pi) times over the original context; it
      keeps f_i where r_i >= beta, takes f_i / s where r_i <= alpha, and the blend
      (1 - gamma) f_i / s + gamma f_i with gamma = (r_i - alpha) / (beta - alpha)
      between. The method's attention temperature is ``yarn_attention_factor``.
    """
    if scaling == "none":
        return rope_inv_freq(D, theta)
    if scaling == "linear":
        return rope_inv_freq(D, theta) / np.float64(factor)
    if scaling == "ntk":
        base = np.float64(theta) * np.power(np.float64(factor), D / (D - 2.0))
        return rope_inv_freq(D, base)
    if scaling == "yarn":
        f = rope_inv_freq(D, theta)
        r = np.float64(original_context) * f / (2.0 * np.pi)
        g = yarn_ramp(r, alpha, beta)
        return (1.0 - g) * f / np.float64(factor) + g * f
    raise ValueError(scaling)


def rope(x: np.ndarray, pos, theta: float, layout: str, inv_freq=None) -> np.ndarray:
    """Rotate the last axis of x at positions ``pos`` (broadcast over x[..., 0]).

    fusedtok README, "Operators" (RoPE, interleaved and NeoX layouts, kv-cache
    pos_offset) and "Usage" (``rope(q, pos_offset=1023, neox=True)``). ``inv_freq``
    (D/2 values) replaces the table theta^(-2i/D) when given: pair i then turns by
    pos * inv_freq[i] (the context-extension tables of ``rope_scaled_inv_freq``).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    f = rope_inv_freq(D, theta) if inv_freq is None else np.asarray(inv_freq, dtype=np.float64)
    if f.shape != (half,):
        raise ValueError(f"inv_freq must hold D/2 = {half} values")
    phi = np.asarray(pos, dtype=np.float64)[..., None] * f
    c, s = np.cos(phi), np.sin(phi)
    if layout == NEOX:
        ia = np.arange(half)
        ib = ia + half
    elif layout == INTERLEAVED:
        ia = 2 * np.arange(half)
        ib = ia + 1
    else:
        raise ValueError(layout)
    a, b = x[..., ia], x[..., ib]
    out = np.empty_like(x)
    out[..., ia] = a * c - b * s
    out[..., ib] = a * s + b * c
    return out


def qknorm_rope(x, norm_w, pos, theta, layout, eps, inv_freq=None):
    """Per-head QK-RMSNorm over D (skipped when norm_w is None), then RoPE at pos[b].

    cutileGPT README, "The current runtime includes" (QK-Norm then RoPE).
    x [B, H, D], pos [B]; ``inv_freq`` as in ``rope``.
    """
    x = np.asarray(x, dtype=np.float64)
    if norm_w is not None:
        x = rms_norm(x, norm_w, eps)
    return rope(x, np.asarray(pos, dtype=np.int64)[:, None], theta, layout, inv_freq)


def qknorm_rope_kv_append(q, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, pos,
                          theta, layout, eps, inv_freq=None):
    """Per-head QK-RMSNorm, RoPE at pos_b, and the K/V append into slot pos_b.

    cutileGPT README, "The current runtime includes" (fused QK-Norm + RoPE +
    KV-cache writes); fusedtok README, "Usage" (caches [B, Hkv, T, D]).
    q [B,Hq,D], k_new/v_new [B,Hkv,D], caches [B,Hkv,T,D], pos [B]; ``inv_freq`` as in
    ``rope``. Returns (rotated q, updated k_cache, updated v_cache); V is stored
    unchanged.
    """
    pos = np.asarray(pos, dtype=np.int64)
    q_out = qknorm_rope(q, q_norm_w, pos, theta, layout, eps, inv_freq)
    k_rot = qknorm_rope(k_new, k_norm_w, pos, theta, layout, eps, inv_freq)
    k_out = np.array(k_cache, dtype=np.float64, copy=True)
    v_out = np.array(v_cache, dtype=np.float64, copy=True)
    for b in range(q_out.shape[0]):
        k_out[b, :, pos[b], :] = k_rot[b]
        v_out[b, :, pos[b], :] = np.asarray(v_new[b], dtype=np.float64)
    return q_out, k_out, v_out


# --------------------------------------------------------------- attention ---
def softmax(z: np.ndarray) -> np.ndarray:
    """Numerically stable softmax over the last axis (fusedtok README, "Operators")."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def default_scale(D: int) -> float:
    return 1.0 / np.sqrt(np.float64(D))


def attend_one(q_h, K, V, scale):
    """softmax(K q * scale) V for one query head over the rows of K and V."""
    if K.shape[0] == 0:
        return np.zeros(np.shape(q_h), dtype=np.float64)
    s = (np.asarray(K, dtype=np.float64) @ np.asarray(q_h, dtype=np.float64)) * scale
    return softmax(s) @ np.asarray(V, dtype=np.float64)


def gqa_decode_attention(q, k_cache, v_cache, lens, scale=None, window=None):
    """Single-query GQA attention over a contiguous cache with per-sequence lengths.

    fusedtok README, "Operators" (attention_decode) and "Usage" (q [B,Hq,D],
    caches [B,Hkv,T,D], lens [B]); "Benchmarks" (heads expanded with
    repeat_interleave). out[b, h] = softmax(q[b,h] . K[b, h//G, lo:len_b] * scale)
    V[b, h//G, lo:len_b], lo = 0, or max(0, len_b - window) with a sliding window
    (cutileGPT README, "The current runtime includes": sliding-window attention; the
    query sees its own token and the window-1 before it).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    scale = default_scale(D) if scale is None else float(scale)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        lo = 0 if window is None else max(0, L - int(window))
        K = np.repeat(np.asarray(k_cache[b, :, lo:L], dtype=np.float64), G, axis=0)  # [Hq, L-lo, D]
        V = np.repeat(np.asarray(v_cache[b, :, lo:L], dtype=np.float64), G, axis=0)
        s = np.einsum("hld,hd->hl", K, q[b]) * scale
        out[b] = np.einsum("hl,hld->hd", softmax(s), V)
    return out


# ------------------------------------------------- split-KV pass and merge ---
def attention_partial(q_h, K, V, scale):
    """One flash-decoding chunk (fusedtok README, "Operators": flash-decoding split).

    For the rows of one chunk: m = max s, l = sum e^(s-m), o = sum e^(s-m) v / l,
    lse = m + ln l. An empty chunk gives o = 0, lse = -inf.
    """
    D = np.shape(q_h)[-1]
    if K.shape[0] == 0:
        return np.zeros(D, dtype=np.float64), -np.inf
    s = (np.asarray(K, dtype=np.float64) @ np.asarray(q_h, dtype=np.float64)) * scale
    m = np.max(s)
    e = np.exp(s - m)
    l = np.sum(e)
    o = (e @ np.asarray(V, dtype=np.float64)) / l
    return o, m + np.log(l)


def merge_partials(os_, lses):
    """Combine chunk results with log-sum-exp weights.

    M = max lse_c; out = sum_c e^(lse_c - M) o_c / sum_c e^(lse_c - M). Chunks with
    lse = -inf carry no weight; with no weighted chunk the result is zero.
    """
    lses = np.asarray(lses, dtype=np.float64)
    os_ = np.asarray(os_, dtype=np.float64)
    if lses.size == 0 or not np.any(np.isfinite(lses)):
        return np.zeros(os_.shape[-1], dtype=np.float64)
    M = np.max(lses)
    w = np.exp(lses - M)
    return np.tensordot(w, os_, axes=(0, 0)) / np.sum(w)


def split_attention(q, k_cache, v_cache, lens, chunks, scale=None):
    """Attention computed as chunk partials then a merge.

    ``chunks`` maps a (b, kv_head) pair to a list of [t0, t1) token ranges that
    partition [0, len_b). Returns (out, partials) with partials[(b, h)] a list of
    (o, lse) in chunk order.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    scale = default_scale(D) if scale is None else float(scale)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    parts = {}
    for b in range(B):
        for h in range(Hq):
            g = h // G
            plist = []
            for (t0, t1) in chunks[(b, g)]:
                K = np.asarray(k_cache[b, g, t0:t1], dtype=np.float64)
                V = np.asarray(v_cache[b, g, t0:t1], dtype=np.float64)
                plist.append(attention_partial(q[b, h], K, V, scale))
            parts[(b, h)] = plist
            if plist:
                out[b, h] = merge_partials([p[0] for p in plist], [p[1] for p in plist])
    return out, parts


# ----------------------------------------------------------- the whole step ---
def decode_step(inp: dict, scale=None):
    """K1 -> K2 -> attention on one step's inputs (all float64).

    ``inp`` keys: x, residual, norm_w, eps, q, k_new, v_new, q_norm_w, k_norm_w,
    k_cache, v_cache, pos, lens, theta, layout, and optionally inv_freq (a RoPE
    frequency table, as in ``rope``). Returns a dict with y, new_residual, q_rot,
    k_cache, v_cache and out.
    """
    y, s = rmsnorm_residual(inp["x"], inp["residual"], inp["norm_w"], inp["eps"])
    q_rot, kc, vc = qknorm_rope_kv_append(inp["q"], inp["k_new"], inp["v_new"],
                                          inp["q_norm_w"], inp["k_norm_w"], inp["k_cache"],
                                          inp["v_cache"], inp["pos"], inp["theta"],
                                          inp["layout"], inp["eps"], inp.get("inv_freq"))
    out = gqa_decode_attention(q_rot, kc, vc, inp["lens"], scale)
    return {"y": y, "new_residual": s, "q_rot": q_rot, "k_cache": kc, "v_cache": vc, "out": out}


# ------------------------------------------- projections on either side of the block ---
def linear(x, w, residual=None):
    """y = x W^T, plus ``residual`` when given.

    x [B, K], w [N, K] (one row per output feature, the weight layout of the
    PyGPUkit 0.2.18 page, "Optimized BF16 GEMV": B[N, K]), residual [B, N]. The
    residual term is the down-projection + residual epilogue of the cutileGPT README,
    "The current runtime includes".
    """
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if residual is not None:
        y = y + residual
    return y


def split_qkv(qkv, Hq, Hkv, D):
    """Cut a packed QKV row block [B, (Hq + 2 Hkv) D] into q [B, Hq, D], k [B, Hkv, D]
    and v [B, Hkv, D] (cutileGPT README, "The current runtime includes": packed QKV
    projections). Reading: the packed columns are all q heads, then all k heads, then
    all v heads, each head's D features contiguous."""
    B = qkv.shape[0]
    q = qkv[:, :Hq * D].reshape(B, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(B, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
    return q, k, v


def attention_sublayer(inp: dict, scale=None, window=None):
    """One decoder layer's attention half around the block, all float64:

        h = x + residual;  y = RMSNorm(h) w;  [q | k | v] = y Wqkv^T;
        q, K/V append = QK-norm + RoPE at pos_b (with ``inv_freq`` when given);  a = attention over the cache;
        out = h + a Wo^T.

    ``inp`` holds the decode_step keys except q, k_new and v_new, plus w_qkv
    [(Hq + 2 Hkv) D, hidden] and w_o [hidden, Hq D]. Returns the intermediates (y,
    h, qkv, q_rot, caches, attn) and ``out``.
    """
    Hq, Hkv, D = inp["Hq"], inp["Hkv"], inp["D"]
    y, h = rmsnorm_residual(inp["x"], inp["residual"], inp["norm_w"], inp["eps"])
    qkv = linear(y, inp["w_qkv"])
    q, k_new, v_new = split_qkv(qkv, Hq, Hkv, D)
    q_rot, kc, vc = qknorm_rope_kv_append(q, k_new, v_new, inp["q_norm_w"], inp["k_norm_w"],
                                          inp["k_cache"], inp["v_cache"], inp["pos"],
                                          inp["theta"], inp["layout"], inp["eps"],
                                          inp.get("inv_freq"))
    attn = gqa_decode_attention(q_rot, kc, vc, inp["lens"], scale, window)
    B = attn.shape[0]
    out = linear(attn.reshape(B, Hq * D), inp["w_o"], h)
    return {"y": y, "h": h, "qkv": qkv, "q_rot": q_rot, "k_cache": kc, "v_cache": vc,
            "attn": attn, "out": out}
