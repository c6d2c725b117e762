"""Scalar brute-force restatement of the block for tiny shapes (test infrastructure only).

Pure-Python loops over nested lists with the ``math`` module, written apart from
the numpy oracle so that a vectorisation or indexing slip in either one (a wrong
axis, a transposed operand, a swapped pair index) shows up as a disagreement on
tiny inputs. Same sources and readings as the numpy oracle: fusedtok 1.0.1 README
("Operators", "Usage") and cutileGPT README ("Why tiles", "The current runtime
includes").
"""
from __future__ import annotations

import math


def rms_norm_row(s, w, eps):
    n = len(s)
    acc = 0.0
    for v in s:
        acc += v * v
    rstd = 1.0 / math.sqrt(acc / n + eps)
    return [s[i] * rstd * w[i] for i in range(n)]


def rmsnorm_residual(x, residual, w, eps):
    ys, ss = [], []
    for r in range(len(x)):
        s = [x[r][i] + (residual[r][i] if residual is not None else 0.0) for i in range(len(x[r]))]
        ss.append(s)
        ys.append(rms_norm_row(s, w, eps))
    return ys, ss


def rope_vec(x, pos, theta, layout, inv_freq=None):
    D = len(x)
    out = list(x)
    for i in range(D // 2):
        inv = theta ** (-(2.0 * i) / D) if inv_freq is None else float(inv_freq[i])
        phi = pos * inv
        c, s = math.cos(phi), math.sin(phi)
        if layout == "neox":
            ia, ib = i, i + D // 2
        else:
            ia, ib = 2 * i, 2 * i + 1
        a, b = x[ia], x[ib]
        out[ia] = a * c - b * s
        out[ib] = a * s + b * c
    return out


def attend(q, K, V, scale):
    """softmax over t of (q . K[t]) * scale, applied to V, by explicit loops."""
    L = len(K)
    D = len(q)
    if L == 0:
        return [0.0] * D
    s = []
    for t in range(L):
        acc = 0.0
        for d in range(D):
            acc += q[d] * K[t][d]
        s.append(acc * scale)
    m = max(s)
    e = [math.exp(v - m) for v in s]
    tot = sum(e)
    out = [0.0] * D
    for t in range(L):
        w = e[t] / tot
        for d in range(D):
            out[d] += w * V[t][d]
    return out


def gqa_decode_attention(q, k_cache, v_cache, lens, scale=None, window=None):
    """q [B][Hq][D], caches [B][Hkv][T][D] as nested lists; query head h reads KV head h // G;
    with a window, only the last `window` tokens of each sequence."""
    B = len(q)
    Hq = len(q[0])
    Hkv = len(k_cache[0])
    G = Hq // Hkv
    D = len(q[0][0])
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = []
    for b in range(B):
        row = []
        for h in range(Hq):
            g = h // G
            L = int(lens[b])
            lo = 0 if window is None else max(0, L - window)
            row.append(attend(q[b][h], k_cache[b][g][lo:L], v_cache[b][g][lo:L], scale))
        out.append(row)
    return out


def linear(x, w, residual=None):
    """y[b][n] = sum_k x[b][k] w[n][k] (+ residual[b][n]), by explicit loops."""
    out = []
    for b in range(len(x)):
        row = []
        for n in range(len(w)):
            acc = 0.0
            for k in range(len(x[b])):
                acc += x[b][k] * w[n][k]
            if residual is not None:
                acc += residual[b][n]
            row.append(acc)
        out.append(row)
    return out


def attention_sublayer(x, residual, norm_w, eps, w_qkv, q_norm_w, k_norm_w, k_cache, v_cache,
                       pos, lens, theta, layout, Hq, Hkv, D, scale=None, window=None):
    """h = x + residual; RMSNorm; packed QKV projection (q heads, then k heads, then v
    heads); QK-norm + RoPE at pos_b; K/V written to slot pos_b; attention; out =
    h + attn W_o^T is left to the caller (returns h and the attention rows)."""
    B = len(x)
    ys, hs = rmsnorm_residual(x, residual, norm_w, eps)
    qkv = linear(ys, w_qkv)
    kc = [[[list(r) for r in k_cache[b][g]] for g in range(Hkv)] for b in range(B)]
    vc = [[[list(r) for r in v_cache[b][g]] for g in range(Hkv)] for b in range(B)]
    q = []
    for b in range(B):
        p = int(pos[b])
        qb = []
        for h in range(Hq):
            v = qkv[b][h * D:(h + 1) * D]
            if q_norm_w is not None:
                v = rms_norm_row(v, q_norm_w, eps)
            qb.append(rope_vec(v, p, theta, layout))
        q.append(qb)
        for g in range(Hkv):
            kv = qkv[b][(Hq + g) * D:(Hq + g + 1) * D]
            vv = qkv[b][(Hq + Hkv + g) * D:(Hq + Hkv + g + 1) * D]
            if k_norm_w is not None:
                kv = rms_norm_row(kv, k_norm_w, eps)
            kc[b][g][p] = rope_vec(kv, p, theta, layout)
            vc[b][g][p] = list(vv)
    attn = gqa_decode_attention(q, kc, vc, lens, scale, window)
    return hs, [sum(attn[b], []) for b in range(B)]


def sample(logits, sampled_ids, penalty, temperature, top_p, top_k, u):
    """The sampler for one row by explicit loops (same readings as the numpy oracle)."""
    z = list(map(float, logits))
    V = len(z)
    seen = []
    for i in sampled_ids:
        i = int(i)
        if 0 <= i < V and i not in seen:
            seen.append(i)
    for i in seen:
        z[i] = z[i] / penalty if z[i] > 0 else z[i] * penalty
    if temperature <= 0:
        best = 0
        for i in range(1, V):
            if z[i] > z[best]:
                best = i
        return best
    z = [v / temperature for v in z]
    m = max(z)
    e = [math.exp(v - m) for v in z]
    tot = sum(e)
    p = [v / tot for v in e]
    # ranking by selection: highest probability first, lower id first among equals
    order, left = [], list(range(V))
    while left:
        best = left[0]
        for i in left[1:]:
            if p[i] > p[best]:
                best = i
        order.append(best)
        left.remove(best)
    n = V if (top_k <= 0 or top_k >= V) else top_k
    kept = order[:n]
    if top_p < 1.0:
        mass = sum(p[i] for i in kept)
        acc, cut = 0.0, []
        for i in kept:
            cut.append(i)
            acc += p[i] / mass
            if acc >= top_p:
                break
        kept = cut
    members = sorted(kept)
    total = sum(p[i] for i in members)
    target = u * total
    acc = 0.0
    for i in members:
        acc += p[i]
        if acc > target:
            return i
    return members[-1]
