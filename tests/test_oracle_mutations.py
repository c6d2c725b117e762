"""Planted mistakes in a copy of the oracle must each fail at least one pin.

The mutants are built here, on the CPU, from the oracle's own functions with one
plausible slip each; the real oracle is never modified.
"""
import inspect
import math
import types

import numpy as np
import pytest

import pins
from oracle import decode_ref as O
from oracle import sampler as SAMPLER


def _sampler_copy(**over):
    """A fresh copy of the sampler module with some functions replaced, so that the
    module's own calls go to the replacements."""
    mod = types.ModuleType("sampler_mutant")
    exec(compile(inspect.getsource(SAMPLER), "sampler_mutant", "exec"), mod.__dict__)
    for name, make in over.items():
        mod.__dict__[name] = make(mod)
    return mod


def _ns(sampler=None, **over):
    d = {k: getattr(O, k) for k in dir(O) if not k.startswith("_")}
    d.update(over)
    d["sampler"] = _sampler_copy(**(sampler or {}))
    return types.SimpleNamespace(**d)


# ---- sampler mutants (each `make(mod)` returns the replacement function)
def _penalty_per_occurrence(mod):
    def f(logits, sampled_ids, penalty):
        z = np.array(logits, dtype=np.float64)
        for i in np.asarray(sampled_ids).ravel():
            i = int(i)
            if 0 <= i < z.size:
                z[i] = z[i] / penalty if z[i] > 0 else z[i] * penalty
        return z
    return f


def _penalty_sign_blind(mod):
    def f(logits, sampled_ids, penalty):
        z = np.array(logits, dtype=np.float64)
        for i in {int(i) for i in np.asarray(sampled_ids).ravel() if 0 <= int(i) < z.size}:
            z[i] = z[i] / penalty
        return z
    return f


def _ties_highest_id(mod):
    def f(p):
        p = np.asarray(p, dtype=np.float64)
        return np.lexsort((-np.arange(p.size), -p))
    return f


def _draw_at_or_above(mod):
    def f(p, keep, u):
        idx = np.nonzero(keep)[0]
        c = np.cumsum(np.asarray(p, dtype=np.float64)[idx])
        j = int(np.searchsorted(c, u * c[-1], side="left"))
        return int(idx[min(j, idx.size - 1)])
    return f


def _top_p_without_renormalising(mod):
    def f(p, top_k=0, top_p=1.0):
        p = np.asarray(p, dtype=np.float64)
        order = mod.ranking(p)
        n = p.size if (top_k <= 0 or top_k >= p.size) else int(top_k)
        kept = order[:n]
        if top_p < 1.0:
            c = np.cumsum(p[kept])
            kept = kept[:min(int(np.searchsorted(c, top_p, side="left")) + 1, n)]
        keep = np.zeros(p.size, dtype=bool)
        keep[kept] = True
        return keep
    return f


def _draw_in_rank_order(mod):
    def f(p, keep, u):
        p = np.asarray(p, dtype=np.float64)
        idx = [i for i in mod.ranking(p) if keep[i]]
        c = np.cumsum(p[idx])
        j = int(np.searchsorted(c, u * c[-1], side="right"))
        return int(idx[min(j, len(idx) - 1)])
    return f


def _greedy_last_max(mod):
    real = mod.sample
    def f(logits, sampled_ids, penalty=1.0, temperature=1.0, top_p=1.0, top_k=0, u=0.0):
        if temperature <= 0:
            z = mod.repetition_penalty(logits, sampled_ids, penalty)
            return int(z.size - 1 - np.argmax(z[::-1]))
        return real(logits, sampled_ids, penalty, temperature, top_p, top_k, u)
    return f


def _rms_eps_outside(s, w, eps):
    s = np.asarray(s, float)
    return s / (np.sqrt(np.mean(s * s, -1, keepdims=True)) + eps) * w


def _rms_sum_not_mean(s, w, eps):
    s = np.asarray(s, float)
    return s / np.sqrt(np.sum(s * s, -1, keepdims=True) + eps) * w


def _rope_factory(sign=1.0, pair="ok", expo=2.0, reverse_table=False):
    def rope(x, pos, theta, layout, inv_freq=None):
        x = np.asarray(x, float)
        D = x.shape[-1]
        half = D // 2
        inv = np.power(float(theta), -expo * np.arange(half) / D)
        if inv_freq is not None:
            inv = np.asarray(inv_freq, float)[::-1] if reverse_table else np.asarray(inv_freq, float)
        phi = np.asarray(pos, float)[..., None] * inv
        c, s = np.cos(phi), np.sin(phi) * sign
        use = layout if pair == "ok" else ("interleaved" if layout == "neox" else "neox")
        if use == "neox":
            ia, ib = np.arange(half), np.arange(half) + half
        else:
            ia, ib = 2 * np.arange(half), 2 * np.arange(half) + 1
        out = np.empty_like(x)
        out[..., ia] = x[..., ia] * c - x[..., ib] * s
        out[..., ib] = x[..., ia] * s + x[..., ib] * c
        return out
    return rope


def _scaled_table_factory(linear_mul=False, ntk_expo=None, ntk_as_linear=False,
                          yarn="ok"):
    def table(D, theta, scaling="none", factor=1.0, original_context=4096, alpha=1.0,
              beta=32.0):
        plain = np.power(float(theta), -2.0 * np.arange(D // 2) / D)
        if scaling == "linear":
            return plain * factor if linear_mul else plain / factor
        if scaling == "ntk":
            if ntk_as_linear:
                return plain / factor
            e = D / (D - 2.0) if ntk_expo is None else ntk_expo(D)
            return np.power(float(theta) * factor ** e, -2.0 * np.arange(D // 2) / D)
        if scaling == "yarn":
            r = original_context * plain / (2 * math.pi)
            if yarn == "ramp_over_index":  # the ramp taken over the pair index instead
                r = np.arange(D // 2)[::-1] * (beta / (D // 2))
            if yarn == "alpha_beta_swapped":
                g = np.clip((r - beta) / (alpha - beta), 0.0, 1.0)
            else:
                g = np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)
            if yarn == "blend_reversed":
                return g * plain / factor + (1 - g) * plain
            return (1 - g) * plain / factor + g * plain
        return plain
    return table


def _attn_factory(group="div", scale_pow=-0.5, transpose_v=False):
    def attn(q, k_cache, v_cache, lens, scale=None, window=None):
        q = np.asarray(q, float)
        B, Hq, D = q.shape
        Hkv = k_cache.shape[1]
        G = Hq // Hkv
        sc = D ** scale_pow if scale is None else scale
        out = np.zeros((B, Hq, D))
        for b in range(B):
            L = int(lens[b])
            for h in range(Hq):
                g = h // G if group == "div" else h % Hkv
                lo = 0 if window is None else max(0, L - window)
                K = np.asarray(k_cache[b, g, lo:L], float)
                V = np.asarray(v_cache[b, g, lo:L], float)
                if L == 0:
                    continue
                p = O.softmax(K @ q[b, h] * sc)
                out[b, h] = (V.T @ p) if not transpose_v else (V[:, :1].T @ p).repeat(D)
        return out
    return attn


def _window_off_by_one(q, k_cache, v_cache, lens, scale=None, window=None):
    if window is not None:
        window = window + 1
    return O.gqa_decode_attention(q, k_cache, v_cache, lens, scale, window)


def _softmax_no_max(z):
    e = np.exp(np.asarray(z, float))
    return e / e.sum(-1, keepdims=True)


def _merge_plain_mean(os_, lses):
    return np.mean(np.asarray(os_, float), axis=0)


def _merge_wrong_sign(os_, lses):
    lses = np.asarray(lses, float)
    w = np.exp(-(lses - np.min(lses)))
    return np.tensordot(w, np.asarray(os_, float), axes=(0, 0)) / w.sum()


def _append_wrong_slot(q, k_new, v_new, qw, kw, kc, vc, pos, theta, layout, eps, inv_freq=None):
    return O.qknorm_rope_kv_append(q, k_new, v_new, qw, kw, kc, vc, np.asarray(pos) + 1 - 1 * (np.asarray(pos) >= kc.shape[2] - 1),
                                   theta, layout, eps, inv_freq)


def _append_norm_after_rope(q, k_new, v_new, qw, kw, kc, vc, pos, theta, layout, eps,
                            inv_freq=None):
    qr = O.rope(np.asarray(q, float), np.asarray(pos)[:, None], theta, layout, inv_freq)
    kr = O.rope(np.asarray(k_new, float), np.asarray(pos)[:, None], theta, layout, inv_freq)
    if qw is not None:
        qr = O.rms_norm(qr, qw, eps)
    if kw is not None:
        kr = O.rms_norm(kr, kw, eps)
    ko, vo = np.array(kc, float), np.array(vc, float)
    for b in range(len(pos)):
        ko[b, :, pos[b]] = kr[b]
        vo[b, :, pos[b]] = v_new[b]
    return qr, ko, vo


def _linear_transposed(x, w, residual=None):
    y = np.asarray(x, float) @ np.asarray(w, float)
    return y if residual is None else y + residual


def _linear_no_residual(x, w, residual=None):
    return np.asarray(x, float) @ np.asarray(w, float).T


def _split_qkv_kv_swapped(qkv, Hq, Hkv, D):
    q, k, v = O.split_qkv(qkv, Hq, Hkv, D)
    return q, v, k


def _sublayer_adds_x(inp, scale=None, window=None):
    res = O.attention_sublayer(inp, scale, window)
    B = res["attn"].shape[0]
    res["out"] = O.linear(res["attn"].reshape(B, -1), inp["w_o"], inp["x"])
    return res


def _margins(mod, unnormalised=False, one_sided=False, shrink=1.0):
    """decision_margins with one slip: the draw margin in unnormalised mass, the top-p
    margin measured on one side of the cut only, or every margin scaled down."""
    real = mod.decision_margins

    def f(logits, sampled_ids, penalty=1.0, temperature=1.0, top_p=1.0, top_k=0, u=0.0):
        m = dict(real(logits, sampled_ids, penalty, temperature, top_p, top_k, u))
        if temperature > 0 and (unnormalised or one_sided):
            p = mod.softmax(mod.repetition_penalty(logits, sampled_ids, penalty) / temperature)
            order = mod.ranking(p)
            n = p.size if (top_k <= 0 or top_k >= p.size) else int(top_k)
            kept = order[:n]
            if one_sided and top_p < 1.0:
                c = np.cumsum(p[kept] / p[kept].sum())
                k = int(np.searchsorted(c, top_p, side="left"))
                m["top_p_cut"] = float(abs(c[min(k, n - 1)] - top_p))
            if unnormalised:
                idx = np.nonzero(mod.nucleus(p, top_k, top_p))[0]
                c = np.cumsum(p[idx])
                j = min(int(np.searchsorted(c, u, side="right")), idx.size - 1)
                lo = c[j - 1] if j > 0 else 0.0
                m["draw"] = float(min(abs(c[j] - u), abs(u - lo)))
        return {k: v * shrink for k, v in m.items()}
    return f


SAMPLER_MUTANTS = {
    "penalty_per_occurrence": dict(repetition_penalty=_penalty_per_occurrence),
    "penalty_ignores_sign": dict(repetition_penalty=_penalty_sign_blind),
    "ties_to_highest_id": dict(ranking=_ties_highest_id),
    "draw_at_or_above_target": dict(draw=_draw_at_or_above),
    "top_p_without_renormalising_top_k": dict(nucleus=_top_p_without_renormalising),
    "draw_in_rank_order": dict(draw=_draw_in_rank_order),
    "greedy_last_maximum": dict(sample=_greedy_last_max),
    "margin_draw_unnormalised": dict(decision_margins=lambda m: _margins(m, unnormalised=True)),
    "margin_top_p_one_sided": dict(decision_margins=lambda m: _margins(m, one_sided=True)),
    "margin_always_small": dict(decision_margins=lambda m: _margins(m, shrink=1e-3)),
}

MUTANTS = {
    "rms_eps_outside_sqrt": dict(rms_norm=_rms_eps_outside,
                                 rmsnorm_residual=lambda x, r, w, e: (_rms_eps_outside(np.asarray(x) + (0 if r is None else np.asarray(r)), w, e), np.asarray(x) + (0 if r is None else np.asarray(r)))),
    "rms_sum_not_mean": dict(rms_norm=_rms_sum_not_mean),
    "rope_sign_flipped": dict(rope=_rope_factory(sign=-1.0)),
    "rope_pairs_swapped": dict(rope=_rope_factory(pair="swapped")),
    "rope_exponent_i_over_d": dict(rope=_rope_factory(expo=1.0)),
    "rope_table_reversed": dict(rope=_rope_factory(reverse_table=True)),
    "rope_linear_multiplies_by_factor": dict(rope_scaled_inv_freq=_scaled_table_factory(linear_mul=True)),
    "rope_ntk_exponent_d_over_d_minus_1": dict(rope_scaled_inv_freq=_scaled_table_factory(ntk_expo=lambda D: D / (D - 1.0))),
    "rope_ntk_scales_every_pair": dict(rope_scaled_inv_freq=_scaled_table_factory(ntk_as_linear=True)),
    "rope_yarn_ramp_over_pair_index": dict(rope_scaled_inv_freq=_scaled_table_factory(yarn="ramp_over_index")),
    "rope_yarn_alpha_beta_swapped": dict(rope_scaled_inv_freq=_scaled_table_factory(yarn="alpha_beta_swapped")),
    "rope_yarn_blend_reversed": dict(rope_scaled_inv_freq=_scaled_table_factory(yarn="blend_reversed")),
    "yarn_factor_log10": dict(yarn_attention_factor=lambda s: 0.1 * math.log10(s) + 1.0 if s > 1 else 1.0),
    "attention_grouping_modulo": dict(gqa_decode_attention=_attn_factory(group="mod")),
    "attention_no_scale": dict(gqa_decode_attention=_attn_factory(scale_pow=0.0)),
    "attention_scale_1_over_d": dict(gqa_decode_attention=_attn_factory(scale_pow=-1.0)),
    "softmax_without_max": dict(softmax=_softmax_no_max),
    "window_one_token_too_many": dict(gqa_decode_attention=_window_off_by_one),
    "merge_plain_mean": dict(merge_partials=_merge_plain_mean),
    "merge_wrong_sign": dict(merge_partials=_merge_wrong_sign),
    "append_norm_after_rope_shared_weight": dict(qknorm_rope_kv_append=_append_norm_after_rope),
    "append_wrong_slot": dict(qknorm_rope_kv_append=_append_wrong_slot),
    "linear_weight_transposed": dict(linear=_linear_transposed),
    "linear_residual_dropped": dict(linear=_linear_no_residual),
    "split_qkv_k_v_swapped": dict(split_qkv=_split_qkv_kv_swapped),
    "sublayer_adds_x_not_h": dict(attention_sublayer=_sublayer_adds_x),
}


@pytest.mark.parametrize("name", sorted(MUTANTS) + sorted(SAMPLER_MUTANTS))
def test_mutant_fails_a_pin(name):
    mutant = _ns(**MUTANTS[name]) if name in MUTANTS else _ns(sampler=SAMPLER_MUTANTS[name])
    failed = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
