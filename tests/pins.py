"""Pins of the CPU oracle: facts the pages and the mathematics fix, stated apart from it.

Each ``pin_*`` takes an oracle-like namespace ``O`` (the real oracle, or a mutant
with one planted mistake) and raises AssertionError when ``O`` disagrees with a
closed form, an invariant, a special case, the hand-derived fixtures in
``golden/closed_forms.json`` or the scalar brute force. ``test_oracle.py`` runs
them against the oracle; ``test_oracle_mutations.py`` checks that plausible
mistakes (a dropped term, a wrong sign or index, a transposed operand) fail at
least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")


def _golden():
    with open(GOLDEN) as f:
        return {c["name"]: c for c in json.load(f)}


def _close(a, b, tol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    same_nan = np.isnan(a) & np.isnan(b)
    err = np.where(same_nan, 0.0, np.abs(a - b))
    scale = np.maximum(1.0, np.where(same_nan, 0.0, np.abs(b)))
    worst = float(np.max(err / scale)) if err.size else 0.0
    assert worst <= tol, f"{what}: relative error {worst:.3e} > {tol:.1e}"


# --------------------------------------------------------------- RMSNorm ---
def pin_rms_unit_rms(O):
    """RMS(y / w) = sqrt(ms / (ms + eps)): unit RMS before the weight, up to eps."""
    rng = np.random.default_rng(1)
    for eps in (1e-6, 0.3):
        s = rng.standard_normal((5, 64)) * 3.0
        w = 1.0 + 0.1 * rng.standard_normal(64)
        y = O.rms_norm(s, w, eps)
        ms = np.mean(s * s, axis=-1)
        _close(np.sqrt(np.mean((y / w) ** 2, axis=-1)), np.sqrt(ms / (ms + eps)), 1e-12, "unit rms")


def pin_rms_constant_row(O):
    """A constant row c gives sign(c) * w / sqrt(1 + eps / c^2)."""
    w = np.linspace(0.5, 1.5, 16)
    for c, eps in ((2.0, 1e-6), (-0.25, 0.01), (7.0, 3.0)):
        y = O.rms_norm(np.full((1, 16), c), w, eps)
        _close(y[0], math.copysign(1.0, c) * w / math.sqrt(1.0 + eps / (c * c)), 1e-13, "const")


def pin_rms_scale_invariance(O):
    """With eps = 0 the norm is invariant to positive scaling and odd in s."""
    rng = np.random.default_rng(2)
    s = rng.standard_normal((3, 32))
    w = rng.standard_normal(32)
    y = O.rms_norm(s, w, 0.0)
    _close(O.rms_norm(s * 37.5, w, 0.0), y, 1e-13, "scale")
    _close(O.rms_norm(-s, w, 0.0), -y, 1e-13, "odd")


def pin_rms_golden(O):
    c = _golden()["rmsnorm_residual_3_4"]
    y, s = O.rmsnorm_residual(np.array(c["x"]), np.array(c["residual"]), np.array(c["w"]), c["eps"])
    _close(y, c["expect_y"], 1e-14, "rms golden y")
    _close(s, c["expect_residual"], 0.0, "rms golden residual")
    y2, s2 = O.rmsnorm_residual(np.array(c["expect_residual"]), None, np.array(c["w"]), c["eps"])
    _close(y2, c["expect_y"], 1e-14, "rms golden without residual")


def pin_rms_brute(O):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 24))
    r = rng.standard_normal((3, 24)) * 2
    w = 1 + 0.1 * rng.standard_normal(24)
    y, s = O.rmsnorm_residual(x, r, w, 1e-6)
    yb, sb = brute.rmsnorm_residual(x.tolist(), r.tolist(), w.tolist(), 1e-6)
    _close(y, yb, 1e-13, "rms brute y")
    _close(s, sb, 0.0, "rms brute residual")


# ------------------------------------------------------------------ RoPE ---
def _pairs(D, layout):
    half = D // 2
    if layout == "neox":
        return np.arange(half), np.arange(half) + half
    return 2 * np.arange(half), 2 * np.arange(half) + 1


def pin_rope_identity_at_zero(O):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 3, 64))
    for layout in ("neox", "interleaved"):
        _close(O.rope(x, np.zeros((2, 3)), 1e4, layout), x, 0.0, "pos 0")


def pin_rope_pair_norms(O):
    """Each declared pair keeps its Euclidean norm at any position."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 128))
    pos = np.array([1, 77, 4095, 131071])
    for layout in ("neox", "interleaved"):
        y = O.rope(x, pos, 5e5, layout)
        ia, ib = _pairs(128, layout)
        _close(np.hypot(y[:, ia], y[:, ib]), np.hypot(x[:, ia], x[:, ib]), 1e-13, "pair norm")


def pin_rope_first_and_last_pair(O):
    """Pair 0 turns by exactly pos radians; the last pair by pos * theta^(-(D-2)/D)."""
    rng = np.random.default_rng(6)
    D, theta = 64, 1e4
    x = rng.standard_normal((3, D))
    pos = np.array([1.0, 1000.0, 131071.0])
    for layout in ("neox", "interleaved"):
        y = O.rope(x, pos, theta, layout)
        ia, ib = _pairs(D, layout)
        for j, ang in ((0, pos), (D // 2 - 1, pos * theta ** (-(D - 2) / D))):
            a, b = x[:, ia[j]], x[:, ib[j]]
            _close(y[:, ia[j]], a * np.cos(ang) - b * np.sin(ang), 1e-12, "pair a")
            _close(y[:, ib[j]], a * np.sin(ang) + b * np.cos(ang), 1e-12, "pair b")


def pin_rope_relative(O):
    """<R(m) q, R(n) k> depends only on m - n."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    for layout in ("neox", "interleaved"):
        a = np.dot(O.rope(q, 500, 1e6, layout), O.rope(k, 120, 1e6, layout))
        b = np.dot(O.rope(q, 1380, 1e6, layout), O.rope(k, 1000, 1e6, layout))
        assert abs(a - b) <= 1e-9 * max(1.0, abs(a)), (layout, a, b)


def pin_rope_layouts_related(O):
    """interleaved(x) = P^-1 neox(P x), where P gathers the even then the odd dims."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 128))
    pos = np.arange(5) * 313.0
    perm = np.concatenate([np.arange(0, 128, 2), np.arange(1, 128, 2)])
    neo = O.rope(x[:, perm], pos, 5e5, "neox")
    back = np.empty_like(neo)
    back[:, perm] = neo
    _close(O.rope(x, pos, 5e5, "interleaved"), back, 1e-13, "layout relation")


def pin_rope_composition(O):
    """R(m) R(n) = R(m + n)."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal(64)
    for layout in ("neox", "interleaved"):
        _close(O.rope(O.rope(x, 300, 1e4, layout), 45, 1e4, layout),
               O.rope(x, 345, 1e4, layout), 1e-12, "composition")


def pin_rope_golden(O):
    g = _golden()
    for name in ("rope_neox_d4", "rope_interleaved_d4"):
        c = g[name]
        _close(O.rope(np.array(c["x"]), c["pos"], c["theta"], c["layout"]), c["expect"], 1e-13, name)


def pin_rope_brute(O):
    rng = np.random.default_rng(10)
    x = rng.standard_normal((3, 16))
    pos = [0, 5, 999]
    for layout in ("neox", "interleaved"):
        y = O.rope(x, np.array(pos), 1e4, layout)
        yb = [brute.rope_vec(x[i].tolist(), pos[i], 1e4, layout) for i in range(3)]
        _close(y, yb, 1e-12, "rope brute")


def pin_rope_table_per_pair(O):
    """With a frequency table given, pair j turns by exactly pos * table[j]."""
    rng = np.random.default_rng(31)
    D = 16
    x = rng.standard_normal((3, D))
    pos = np.array([0.0, 7.0, 40000.0])
    table = rng.uniform(0.0, 1.0, D // 2)
    table[3] = 0.0  # a pair that does not turn
    for layout in ("neox", "interleaved"):
        y = O.rope(x, pos, 1e4, layout, inv_freq=table)
        ia, ib = _pairs(D, layout)
        for j in range(D // 2):
            ang = pos * table[j]
            a, b = x[:, ia[j]], x[:, ib[j]]
            _close(y[:, ia[j]], a * np.cos(ang) - b * np.sin(ang), 1e-11, "table pair a")
            _close(y[:, ib[j]], a * np.sin(ang) + b * np.cos(ang), 1e-11, "table pair b")
        yb = [brute.rope_vec(x[i].tolist(), pos[i], 1e4, layout, table) for i in range(3)]
        _close(y, yb, 1e-12, "table brute")


def pin_rope_linear_interpolation(O):
    """Linear position interpolation by s: the rotation at position s * p with the
    scaled table is the plain rotation at p, and every frequency is the plain one / s."""
    rng = np.random.default_rng(32)
    D, theta = 128, 5e5
    x = rng.standard_normal((4, D))
    p = np.array([1.0, 333.0, 8191.0, 32767.0])
    slowest = theta ** (-(D - 2) / D)
    for s in (2.0, 4.0, 8.0):
        t = O.rope_scaled_inv_freq(D, theta, "linear", s)
        assert t.shape == (D // 2,)
        assert abs(t[0] - 1.0 / s) <= 1e-15, t[0]
        assert abs(t[-1] * s / slowest - 1.0) <= 1e-13, t[-1]
        for layout in ("neox", "interleaved"):
            _close(O.rope(x, s * p, theta, layout, inv_freq=t), O.rope(x, p, theta, layout),
                   1e-9, "linear interpolation")


def pin_rope_ntk_table(O):
    """NTK-aware base change by s: pair 0 keeps frequency 1, the slowest pair turns
    exactly s times slower than in the plain table, consecutive frequencies keep one
    common ratio (the table is a plain table of some base), and s = 1, like the
    unscaled table, gives theta^(-2i/D)."""
    for D, theta in ((64, 1e4), (128, 5e5), (128, 1e6)):
        plain = theta ** (-2.0 * np.arange(D // 2) / D)
        for s in (2.0, 4.0, 16.0):
            t = O.rope_scaled_inv_freq(D, theta, "ntk", s)
            assert t.shape == (D // 2,)
            assert t[0] == 1.0, t[0]
            assert abs(t[-1] * s / plain[-1] - 1.0) <= 1e-12, (D, s, t[-1])
            r = t[1:] / t[:-1]
            assert np.max(np.abs(r / r[0] - 1.0)) <= 1e-12, (D, s)
        _close(O.rope_scaled_inv_freq(D, theta, "ntk", 1.0), plain, 1e-14, "ntk s=1")
        _close(O.rope_scaled_inv_freq(D, theta, "none", 7.0), plain, 1e-14, "unscaled")
    # D = 4: the base grows by s^2, so the second pair turns at theta^-1/2 / s
    t = O.rope_scaled_inv_freq(4, 1e4, "ntk", 4.0)
    _close(t, [1.0, 0.0025], 1e-15, "ntk D=4")


def pin_rope_yarn_table(O):
    """YaRN: a pair that turns at least beta times over the original context keeps its
    plain frequency f, one that turns at most alpha times gets f / s, and between them
    the share of f it keeps, (t / f - 1/s) / (1 - 1/s), grows linearly with the number
    of turns r = L f / (2 pi), from 0 at alpha to 1 at beta. s = 1 gives the plain
    table; the attention factor 0.1 ln(s) + 1 is 1.1 at s = e and 2 at s = e^10."""
    for D, theta, L, s in ((128, 5e5, 8192, 8.0), (64, 1e4, 2048, 4.0), (128, 1e6, 4096, 16.0)):
        f = theta ** (-2.0 * np.arange(D // 2) / D)
        r = L * f / (2.0 * math.pi)
        t = O.rope_scaled_inv_freq(D, theta, "yarn", s, L, 1.0, 32.0)
        keep = (t / f - 1.0 / s) / (1.0 - 1.0 / s)
        assert np.all(np.abs(keep[r >= 32.0] - 1.0) <= 1e-12), (D, "fast pairs")
        assert np.all(np.abs(keep[r <= 1.0]) <= 1e-12), (D, "slow pairs")
        mid = (r > 1.0) & (r < 32.0)
        assert mid.sum() >= 3, (D, int(mid.sum()))
        slope, icpt = np.polyfit(r[mid], keep[mid], 1)
        assert abs(slope - 1.0 / 31.0) <= 1e-10 and abs(icpt + 1.0 / 31.0) <= 1e-9, (slope, icpt)
        _close(O.rope_scaled_inv_freq(D, theta, "yarn", 1.0, L), f, 1e-14, "yarn s=1")
    assert O.yarn_attention_factor(1.0) == 1.0
    _close(O.yarn_attention_factor(math.e), 1.1, 1e-15, "factor at e")
    _close(O.yarn_attention_factor(math.e ** 10), 2.0, 1e-15, "factor at e^10")


# ---------------------------------------------------- QK-norm and append ---
def pin_append_golden(O):
    c = _golden()["qknorm_rope_append_d4"]
    q, kc, vc = O.qknorm_rope_kv_append(
        np.array(c["q"]), np.array(c["k_new"]), np.array(c["v_new"]), np.array(c["q_norm_w"]),
        np.array(c["k_norm_w"]), np.array(c["k_cache"]), np.array(c["v_cache"]),
        np.array(c["pos"]), c["theta"], c["layout"], c["eps"])
    _close(q, c["expect_q"], 1e-13, "append q")
    _close(kc, c["expect_k_cache"], 1e-13, "append k cache")
    _close(vc, c["expect_v_cache"], 0.0, "append v cache")


def pin_append_slots(O):
    """Only slot pos_b changes; V lands bit for bit; with QK-norm the rotated head has unit RMS."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, T, D = 3, 4, 2, 9, 32
    q = rng.standard_normal((B, Hq, D))
    kn = rng.standard_normal((B, Hkv, D))
    vn = rng.standard_normal((B, Hkv, D))
    kc = rng.standard_normal((B, Hkv, T, D))
    vc = rng.standard_normal((B, Hkv, T, D))
    kc[:, :, 6:] = np.nan
    vc[:, :, 6:] = np.nan
    pos = np.array([0, 3, 8])
    ones = np.ones(D)
    qo, ko, vo = O.qknorm_rope_kv_append(q, kn, vn, ones, ones, kc, vc, pos, 1e4, "neox", 0.0)
    for b in range(B):
        mask = np.ones(T, bool)
        mask[pos[b]] = False
        _close(ko[b][:, mask], kc[b][:, mask], 0.0, "other k slots")
        _close(vo[b][:, mask], vc[b][:, mask], 0.0, "other v slots")
        _close(vo[b, :, pos[b]], vn[b], 0.0, "v slot")
    _close(np.sqrt(np.mean(qo ** 2, -1)), np.ones((B, Hq)), 1e-13, "q unit rms")
    _close(np.sqrt(np.mean(ko[np.arange(B), :, pos] ** 2, -1)), np.ones((B, Hkv)), 1e-13, "k unit rms")
    # pos 0: no rotation, so the stored key is the normalised new key itself
    _close(ko[0, :, 0], kn[0] / np.sqrt(np.mean(kn[0] ** 2, -1, keepdims=True)), 1e-13, "k at pos 0")
    # without QK-norm and at pos 0, q passes through
    qo2, _, _ = O.qknorm_rope_kv_append(q, kn, vn, None, None, kc, vc, np.zeros(B, int),
                                        1e4, "interleaved", 1e-6)
    _close(qo2, q, 0.0, "q passthrough")


# ---------------------------------------------------------------- softmax ---
def pin_softmax_stable(O):
    rng = np.random.default_rng(12)
    z = rng.standard_normal((4, 50)) * 5
    p = O.softmax(z)
    _close(p.sum(-1), np.ones(4), 1e-14, "sums to one")
    _close(O.softmax(z + 1e4), p, 1e-12, "shift 1e4")
    assert np.all(np.isfinite(O.softmax(np.array([1e4, 1e4 - 1.0, -1e4])))), "overflow"


# -------------------------------------------------------------- attention ---
def pin_attention_golden(O):
    c = _golden()["attention_two_keys"]
    out = O.gqa_decode_attention(np.array(c["q"]), np.array(c["k_cache"]), np.array(c["v_cache"]),
                                 np.array(c["lens"]))
    _close(out, c["expect"], 1e-13, "attention golden")


def pin_attention_special_cases(O):
    rng = np.random.default_rng(13)
    B, Hq, Hkv, T, D = 2, 8, 2, 40, 16
    q = rng.standard_normal((B, Hq, D)) * 3
    kc = rng.standard_normal((B, Hkv, T, D))
    vc = rng.standard_normal((B, Hkv, T, D))
    lens = np.array([1, 30])
    kc[0, :, 1:] = np.nan
    vc[0, :, 1:] = np.nan
    kc[1, :, 30:] = np.nan
    vc[1, :, 30:] = np.nan
    out = O.gqa_decode_attention(q, kc, vc, lens)
    G = Hq // Hkv
    # one key: the output is that key's value, whatever q is
    _close(out[0], np.repeat(vc[0, :, 0], G, axis=0), 1e-13, "single key")
    # identical keys: the mean of V
    kc2 = kc.copy()
    kc2[1, :, :30] = kc[1, :, :1]
    out2 = O.gqa_decode_attention(q, kc2, vc, lens)
    _close(out2[1], np.repeat(vc[1, :, :30].mean(1), G, axis=0), 1e-12, "identical keys")
    # q = 0: the mean of V
    out3 = O.gqa_decode_attention(np.zeros_like(q), kc, vc, lens)
    _close(out3[1], np.repeat(vc[1, :, :30].mean(1), G, axis=0), 1e-12, "zero query")
    assert np.all(np.isfinite(out)), "NaN past len leaked into the output"
    # length 0 yields zeros
    out4 = O.gqa_decode_attention(q, kc, vc, np.array([0, 30]))
    _close(out4[0], np.zeros((Hq, D)), 0.0, "empty")


def pin_attention_grouping(O):
    """Query head h reads KV head h // G: give each KV head one distinct key/value."""
    B, Hq, Hkv, D = 1, 12, 3, 8
    G = Hq // Hkv
    kc = np.zeros((B, Hkv, 2, D))
    vc = np.zeros((B, Hkv, 2, D))
    for g in range(Hkv):
        kc[0, g, 0] = g + 1.0
        vc[0, g, 0] = 10.0 * (g + 1) + np.arange(D)
    kc[0, :, 1] = np.nan
    vc[0, :, 1] = np.nan
    q = np.random.default_rng(14).standard_normal((B, Hq, D))
    out = O.gqa_decode_attention(q, kc, vc, np.array([1]))
    for h in range(Hq):
        _close(out[0, h], vc[0, h // G, 0], 0.0, f"head {h}")


def pin_attention_scale(O):
    """Two keys with logit gap a: the first weight is the logistic of a (scale 1/sqrt(D))."""
    D = 16
    a = 1.7
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = a * math.sqrt(D)
    kc = np.zeros((1, 1, 2, D))
    kc[0, 0, 0, 0] = 1.0
    vc = np.zeros((1, 1, 2, D))
    vc[0, 0, 0, 1] = 1.0
    vc[0, 0, 1, 2] = 1.0
    out = O.gqa_decode_attention(q, kc, vc, np.array([2]))
    w0 = 1.0 / (1.0 + math.exp(-a))
    _close(out[0, 0, 1:3], [w0, 1.0 - w0], 1e-14, "scale")
    out2 = O.gqa_decode_attention(q, kc, vc, np.array([2]), scale=0.0)
    _close(out2[0, 0, 1:3], [0.5, 0.5], 1e-14, "explicit scale")


def pin_attention_brute(O):
    rng = np.random.default_rng(15)
    B, Hq, Hkv, T, D = 2, 6, 3, 7, 8
    q = rng.standard_normal((B, Hq, D)) * 2
    kc = rng.standard_normal((B, Hkv, T, D))
    vc = rng.standard_normal((B, Hkv, T, D))
    lens = np.array([7, 3])
    out = O.gqa_decode_attention(q, kc, vc, lens)
    ref = brute.gqa_decode_attention(q.tolist(), kc.tolist(), vc.tolist(), lens.tolist())
    _close(out, ref, 1e-12, "attention brute")


def pin_attention_window(O):
    """Sliding window: window >= len is plain attention, window 1 returns the newest
    token's value, and a window equals plain attention on the cache cut to its rows."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, T, D = 3, 4, 2, 30, 8
    q = rng.standard_normal((B, Hq, D)) * 2
    kc = rng.standard_normal((B, Hkv, T, D))
    vc = rng.standard_normal((B, Hkv, T, D))
    lens = np.array([30, 5, 12])
    full = O.gqa_decode_attention(q, kc, vc, lens)
    _close(O.gqa_decode_attention(q, kc, vc, lens, window=30), full, 1e-14, "window >= len")
    one = O.gqa_decode_attention(q, kc, vc, lens, window=1)
    for b in range(B):
        _close(one[b], np.repeat(vc[b, :, lens[b] - 1], Hq // Hkv, axis=0), 1e-14, "window 1")
    W = 7
    for b in range(B):
        lo = max(0, lens[b] - W)
        cut = O.gqa_decode_attention(q[b:b + 1], kc[b:b + 1, :, lo:lens[b]], vc[b:b + 1, :, lo:lens[b]],
                                     np.array([lens[b] - lo]))
        _close(O.gqa_decode_attention(q, kc, vc, lens, window=W)[b], cut[0], 1e-13, "window cut")
    ref = brute.gqa_decode_attention(q.tolist(), kc.tolist(), vc.tolist(), lens.tolist(), window=W)
    _close(O.gqa_decode_attention(q, kc, vc, lens, window=W), ref, 1e-12, "window brute")



# -------------------------------------------------------- projections ---
def pin_linear_one_hot(O):
    """x = e_k gives column k of W; W = I gives x back; W = 0 gives the residual."""
    rng = np.random.default_rng(21)
    N, K = 5, 3
    w = rng.standard_normal((N, K))
    y = O.linear(np.eye(K), w)
    _close(y, w.T, 1e-15, "one-hot rows pick columns of W")
    x = rng.standard_normal((4, K))
    _close(O.linear(x, np.eye(K)), x, 1e-15, "identity weight")
    r = rng.standard_normal((4, N))
    _close(O.linear(x, np.zeros((N, K)), r), r, 1e-15, "zero weight keeps the residual")
    _close(O.linear(x, w, r) - O.linear(x, w), r, 1e-13, "residual added once")


def pin_linear_brute(O):
    rng = np.random.default_rng(22)
    x = rng.standard_normal((3, 7))
    w = rng.standard_normal((11, 7))
    r = rng.standard_normal((3, 11))
    _close(O.linear(x, w, r), brute.linear(x.tolist(), w.tolist(), r.tolist()), 1e-12, "linear brute")
    _close(O.linear(x, w), brute.linear(x.tolist(), w.tolist()), 1e-12, "linear brute, no residual")


def pin_split_qkv_order(O):
    """Packed columns: every q head, then every k head, then every v head."""
    Hq, Hkv, D, B = 4, 2, 3, 2
    qkv = np.arange(B * (Hq + 2 * Hkv) * D, dtype=np.float64).reshape(B, -1)
    q, k, v = O.split_qkv(qkv, Hq, Hkv, D)
    row = (Hq + 2 * Hkv) * D
    for b in range(B):
        for h in range(Hq):
            _close(q[b, h], b * row + h * D + np.arange(D), 0, "q head columns")
        for g in range(Hkv):
            _close(k[b, g], b * row + (Hq + g) * D + np.arange(D), 0, "k head columns")
            _close(v[b, g], b * row + (Hq + Hkv + g) * D + np.arange(D), 0, "v head columns")


def _sublayer_inputs(rng, B=2, Hq=4, Hkv=2, D=8, T=9, hidden=None, qk_norm=True):
    hidden = Hq * D if hidden is None else hidden
    pos = np.array([T - 1, 3])[:B]
    inp = dict(
        x=rng.standard_normal((B, hidden)), residual=rng.standard_normal((B, hidden)),
        norm_w=1 + 0.1 * rng.standard_normal(hidden), eps=1e-6,
        w_qkv=rng.standard_normal(((Hq + 2 * Hkv) * D, hidden)) / math.sqrt(hidden),
        w_o=rng.standard_normal((hidden, Hq * D)) / math.sqrt(Hq * D),
        q_norm_w=(1 + 0.1 * rng.standard_normal(D)) if qk_norm else None,
        k_norm_w=(1 + 0.1 * rng.standard_normal(D)) if qk_norm else None,
        k_cache=rng.standard_normal((B, Hkv, T, D)), v_cache=rng.standard_normal((B, Hkv, T, D)),
        pos=pos, lens=pos + 1, theta=1e4, layout="interleaved", Hq=Hq, Hkv=Hkv, D=D)
    return inp


def pin_sublayer_reduces_to_block(O):
    """With a selection matrix for Wqkv the sublayer is the pinned block fed with the
    selected features; with Wo = 0 the output is the residual stream h, and with
    Wo = I it is h plus the attention rows."""
    rng = np.random.default_rng(23)
    Hq, Hkv, D = 4, 2, 8
    inp = _sublayer_inputs(rng, Hq=Hq, Hkv=Hkv, D=D)
    hidden = Hq * D
    sel = rng.permutation(hidden)
    ksel, vsel = sel[:Hkv * D], sel[hidden - Hkv * D:]
    w_qkv = np.zeros(((Hq + 2 * Hkv) * D, hidden))
    w_qkv[np.arange(hidden), np.arange(hidden)] = 1.0
    w_qkv[hidden + np.arange(Hkv * D), ksel] = 1.0
    w_qkv[hidden + Hkv * D + np.arange(Hkv * D), vsel] = 1.0
    for w_o, with_attn in ((np.zeros((hidden, hidden)), False), (np.eye(hidden), True)):
        run = dict(inp, w_qkv=w_qkv, w_o=w_o)
        res = O.attention_sublayer(run)
        h = inp["x"] + inp["residual"]
        y = O.rms_norm(h, inp["norm_w"], inp["eps"])
        B = h.shape[0]
        blk = O.decode_step(dict(inp, q=y.reshape(B, Hq, D), k_new=y[:, ksel].reshape(B, Hkv, D),
                                 v_new=y[:, vsel].reshape(B, Hkv, D)))
        _close(res["h"], h, 1e-14, "sublayer residual stream")
        _close(res["k_cache"], blk["k_cache"], 1e-13, "sublayer K append")
        _close(res["v_cache"], blk["v_cache"], 1e-13, "sublayer V append")
        expect = h + (blk["out"].reshape(B, hidden) if with_attn else 0.0)
        _close(res["out"], expect, 1e-12, "sublayer output")


def pin_sublayer_brute(O):
    rng = np.random.default_rng(24)
    for qk_norm, layout in ((True, "interleaved"), (False, "neox")):
        inp = _sublayer_inputs(rng, B=2, Hq=4, Hkv=2, D=4, T=6, hidden=12, qk_norm=qk_norm)
        inp["layout"] = layout
        res = O.attention_sublayer(inp, window=4)
        L = lambda a: None if a is None else np.asarray(a).tolist()
        hs, attn = brute.attention_sublayer(
            L(inp["x"]), L(inp["residual"]), L(inp["norm_w"]), inp["eps"], L(inp["w_qkv"]),
            L(inp["q_norm_w"]), L(inp["k_norm_w"]), L(inp["k_cache"]), L(inp["v_cache"]),
            L(inp["pos"]), L(inp["lens"]), inp["theta"], layout, 4, 2, 4, window=4)
        out = brute.linear(attn, L(inp["w_o"]), hs)
        _close(res["out"], out, 1e-12, f"sublayer brute {layout}")

# ---------------------------------------------------------- split + merge ---
def pin_merge_golden(O):
    c = _golden()["merge_two_chunks"]
    _close(O.merge_partials(np.array(c["o"]), np.array(c["lse"])), c["expect"], 1e-15, "merge golden")


def pin_split_equals_unsplit(O):
    """Any partition of [0, len) merged by log-sum-exp equals unsplit attention."""
    rng = np.random.default_rng(16)
    B, Hq, Hkv, T, D = 2, 4, 2, 50, 16
    q = rng.standard_normal((B, Hq, D)) * 2
    kc = rng.standard_normal((B, Hkv, T, D))
    vc = rng.standard_normal((B, Hkv, T, D))
    kc[:, :, :, 0] *= 6.0
    lens = np.array([50, 17])
    ref = O.gqa_decode_attention(q, kc, vc, lens)
    for trial in range(4):
        chunks = {}
        for b in range(B):
            for g in range(Hkv):
                cuts = sorted(set(rng.integers(0, lens[b] + 1, size=trial + 1).tolist()) | {0, int(lens[b])})
                chunks[(b, g)] = list(zip(cuts[:-1], cuts[1:]))
                if trial == 3:  # empty chunks carry lse = -inf and no weight
                    chunks[(b, g)] = [(0, 0)] + chunks[(b, g)] + [(int(lens[b]), int(lens[b]))]
        out, parts = O.split_attention(q, kc, vc, lens, chunks)
        _close(out, ref, 1e-12, f"split trial {trial}")
        # the same through the pieces: one partial per chunk, then the merge
        G = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                ps = [O.attention_partial(q[b, h], kc[b, h // G, t0:t1], vc[b, h // G, t0:t1], 0.25)
                      for (t0, t1) in chunks[(b, h // G)]]
                _close(O.merge_partials([p[0] for p in ps], [p[1] for p in ps]), ref[b, h], 1e-12,
                       "partials merged")
    # a single chunk: the partial itself is the answer and lse is log sum exp of the logits
    o, lse = O.attention_partial(q[0, 0], kc[0, 0, :50], vc[0, 0, :50], 0.25)
    s = kc[0, 0, :50] @ q[0, 0] * 0.25
    assert abs(lse - (np.max(s) + math.log(np.sum(np.exp(s - np.max(s)))))) <= 1e-12
    _close(o, O.gqa_decode_attention(q, kc, vc, lens)[0, 0], 1e-12, "single chunk")



# ------------------------------------------------------------- sampler ---
def _S(O):
    return O.sampler if hasattr(O, "sampler") else O


def pin_penalty_ctrl(O):
    """CTRL: positive logits divided, negative (and zero) multiplied, each distinct id
    in range once; padding and out-of-range ids ignored."""
    S = _S(O)
    z = S.repetition_penalty([2.0, -2.0, 0.0, 3.0, 5.0], [0, 1, 1, 7, -1, 4, 4, 4], 2.0)
    _close(z, [1.0, -4.0, 0.0, 3.0, 2.5], 0, "penalty")
    _close(S.repetition_penalty([1.5, -0.5], [0, 1], 1.0), [1.5, -0.5], 0, "penalty 1")


def pin_greedy(O):
    S = _S(O)
    assert S.sample([1.0, 3.0, 3.0, 2.0], [], 1.0, 0.0) == 1  # first of the tied maxima
    assert S.sample([1.0, 3.0, 2.9, 2.0], [1], 2.0, 0.0) == 2  # penalty moves the argmax
    for u in (0.0, 0.5, 0.999):
        assert S.sample([0.1, 0.7, 0.2], [], 1.0, 1e-4, u=u) == 1  # T -> 0 is greedy


def pin_draw_inverse_cdf(O):
    """With exact binary masses the token boundaries are exact: token i for
    u in [c_{i-1}, c_i) in token-id order, the boundary itself going up."""
    S = _S(O)
    p = np.array([0.125, 0.125, 0.25, 0.5])
    keep = np.ones(4, dtype=bool)
    for u, tok in ((0.0, 0), (0.1249, 0), (0.125, 1), (0.2499, 1), (0.25, 2), (0.4999, 2),
                   (0.5, 3), (0.9999, 3)):
        assert S.draw(p, keep, u) == tok, (u, tok)
    keep = np.array([False, True, False, True])  # nucleus {1, 3}: masses 1/8, 1/2 -> 1/5, 4/5
    for u, tok in ((0.0, 1), (0.1999, 1), (0.2, 3), (0.99, 3)):
        assert S.draw(p, keep, u) == tok, (u, tok)


def pin_topk_topp_closed_form(O):
    """probabilities 0.1, 0.2, 0.3, 0.4 (logits log 1..4): the ranking is 3, 2, 1, 0."""
    S = _S(O)
    z = np.log([1.0, 2.0, 3.0, 4.0])
    p = S.softmax(z)
    _close(p, [0.1, 0.2, 0.3, 0.4], 1e-15, "softmax")
    assert list(S.ranking(p)) == [3, 2, 1, 0]
    assert list(np.nonzero(S.nucleus(p, 0, 0.65))[0]) == [2, 3]      # 0.4 + 0.3 >= 0.65
    assert list(np.nonzero(S.nucleus(p, 0, 0.71))[0]) == [1, 2, 3]   # needs the 0.2
    assert list(np.nonzero(S.nucleus(p, 0, 0.05))[0]) == [3]         # the top token alone
    assert list(np.nonzero(S.nucleus(p, 1, 1.0))[0]) == [3]
    assert list(np.nonzero(S.nucleus(p, 3, 1.0))[0]) == [1, 2, 3]
    # top-k renormalises before top-p: within {3, 2} the masses are 4/7 and 3/7
    assert list(np.nonzero(S.nucleus(p, 2, 0.56))[0]) == [3]
    assert list(np.nonzero(S.nucleus(p, 2, 0.58))[0]) == [2, 3]
    # sample: nucleus {2, 3} in id order, masses 3/7 then 4/7
    assert S.sample(z, [], 1.0, 1.0, 0.65, 0, u=0.42) == 2
    assert S.sample(z, [], 1.0, 1.0, 0.65, 0, u=0.43) == 3
    # temperature 0.5 squares the odds: 1, 4, 9, 16 (sum 30)
    _close(S.softmax(z / 0.5), np.array([1, 4, 9, 16]) / 30.0, 1e-14, "temperature")


def pin_ties_by_lowest_id(O):
    S = _S(O)
    p = S.softmax([1.0, 2.0, 2.0, 2.0, 0.0])
    assert list(S.ranking(p)) == [1, 2, 3, 0, 4]
    assert list(np.nonzero(S.nucleus(p, 2, 1.0))[0]) == [1, 2]


def pin_sampler_distribution(O):
    """Over a fine grid of u the draw reproduces the renormalised nucleus exactly."""
    S = _S(O)
    rng = np.random.default_rng(31)
    z = rng.standard_normal(20) * 1.5
    ids = [3, 3, 17, 25, -1]
    zp = S.repetition_penalty(z, ids, 1.4)
    p = S.softmax(zp / 0.8)
    keep = S.nucleus(p, 7, 0.8)
    q = np.where(keep, p, 0.0)
    q /= q.sum()
    n = 20000
    counts = np.zeros(20)
    for j in range(n):
        counts[S.sample(z, ids, 1.4, 0.8, 0.8, 7, u=(j + 0.5) / n)] += 1
    assert np.max(np.abs(counts / n - q)) <= 1.0 / n + 1e-12
    # the nucleus is the shortest mass-p prefix of the top-7 ranking
    order = S.ranking(p)[:7]
    kept = [i for i in order if keep[i]]
    assert kept == list(order[:len(kept)])
    mass = p[order].sum()
    assert p[kept].sum() / mass >= 0.8 and p[kept[:-1]].sum() / mass < 0.8


def pin_decision_margins(O):
    """The margins that decide when a GPU token may differ from the oracle's, derived by
    hand on probabilities 0.1, 0.2, 0.3, 0.4 (logits log 1..4; ranking 3, 2, 1, 0;
    renormalised prefix masses 0.4, 0.7, 0.9, 1), then checked as what they claim to be:
    moving u (or top_p) by less than the margin keeps the token, by a little more flips it."""
    S = _S(O)
    z = np.log([1.0, 2.0, 3.0, 4.0])
    # top-p 0.65: the cut falls after 0.7, 0.05 above p and 0.25 past the 0.4 before it;
    # nucleus {2, 3} in id order has running masses 3/7, 1; u = 0.42 is 3/7 - 0.42 below 3/7
    m = S.decision_margins(z, [], 1.0, 1.0, 0.65, 0, 0.42)
    _close([m["top_p_cut"], m["draw"]], [0.05, 3.0 / 7.0 - 0.42], 1e-12, "margins p=0.65")
    m = S.decision_margins(z, [], 1.0, 1.0, 0.65, 0, 0.9)  # 0.1 below the end, 0.47 above 3/7
    _close([m["draw"]], [0.1], 1e-12, "draw margin u=0.9")
    # top-p 0.71: 0.01 past the 0.7 prefix; nucleus {1, 2, 3}: running masses 2/9, 5/9, 1
    m = S.decision_margins(z, [], 1.0, 1.0, 0.71, 0, 0.5)
    _close([m["top_p_cut"], m["draw"]], [0.01, 1.0 / 18.0], 1e-12, "margins p=0.71")
    # top-k 2 renormalises to 4/7, 3/7: p = 0.56 is 4/7 - 0.56 below the first prefix
    m = S.decision_margins(z, [], 1.0, 1.0, 0.56, 2, 0.3)
    _close([m["top_p_cut"], m["draw"]], [4.0 / 7.0 - 0.56, 0.3], 1e-12, "margins k=2")
    assert S.decision_margins(z, [], 1.0, 1.0, 1.0, 0, 0.3)["top_p_cut"] == np.inf
    # greedy: the gap between the two largest penalised logits
    _close([S.decision_margins([1.0, 3.0, 2.9, 2.0], [], 1.0, 0.0)["argmax_gap"]], [0.1], 1e-12, "gap")
    _close([S.decision_margins([1.0, 3.0, 2.9, 2.0], [1], 2.0, 0.0)["argmax_gap"]], [0.9], 1e-12,
           "gap after the penalty")
    # the margins are the distances to the nearest boundary
    rng = np.random.default_rng(33)
    checked = 0
    for _ in range(60):
        V = int(rng.integers(3, 12))
        zz = rng.standard_normal(V) * 1.5
        T, tp, tk, u = 0.9, float(rng.choice([0.5, 0.8, 0.95])), int(rng.choice([0, 4])), float(rng.random())
        m = S.decision_margins(zz, [], 1.0, T, tp, tk, u)
        tok = S.sample(zz, [], 1.0, T, tp, tk, u)
        d = m["draw"]
        for uu in (u - 0.99 * d, u + 0.99 * d):
            if 0.0 <= uu < 1.0:
                assert S.sample(zz, [], 1.0, T, tp, tk, uu) == tok
        # with both sides inside [0, 1) the nearest boundary is an interior one (the
        # ends 0 and 1 count as boundaries too, which only makes a margin smaller)
        if 0.0 <= u - 1.01 * d and u + 1.01 * d < 1.0:
            assert any(S.sample(zz, [], 1.0, T, tp, tk, uu) != tok
                       for uu in (u - 1.01 * d, u + 1.01 * d)), "a boundary closer than the margin"
            checked += 1
        c = m["top_p_cut"]
        p = S.softmax(zz / T)
        keep = S.nucleus(p, tk, tp)
        for pp in (tp - 0.99 * c, tp + 0.99 * c):
            if 0.0 < pp < 1.0:
                assert np.array_equal(S.nucleus(p, tk, pp), keep)
        if 0.0 < tp - 1.01 * c and tp + 1.01 * c < 1.0:
            assert any(not np.array_equal(S.nucleus(p, tk, pp), keep)
                       for pp in (tp - 1.01 * c, tp + 1.01 * c)), "a cut closer than the margin"
            checked += 1
    assert checked >= 40


def pin_sampler_brute(O):
    S = _S(O)
    rng = np.random.default_rng(32)
    for t in range(150):
        V = int(rng.integers(2, 25))
        z = rng.standard_normal(V) * 2
        if t % 3 == 0:
            z = np.round(z)  # ties
        ids = rng.integers(-2, V + 2, size=6)
        args = (float(rng.choice([1.0, 1.3, 2.0])), float(rng.choice([0.0, 0.6, 1.0])),
                float(rng.choice([1.0, 0.9, 0.4])), int(rng.choice([0, 1, 3, V])),
                float(rng.random()))
        m = S.decision_margins(z, ids, *args)
        if min(m.values()) < 1e-9:
            continue
        assert S.sample(z, ids, *args) == brute.sample(z.tolist(), ids.tolist(), *args), (t, args)

ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
