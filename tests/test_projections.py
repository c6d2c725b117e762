"""Projections around the block and the attention sublayer, CUDA path against the
CPU oracle on identical seeded bf16 inputs (GPU only).

The projection is checked element by element over shapes that span one and many
128-feature tiles, every batch tile size (16 .. 256 rows) with a ragged last tile,
split and unsplit K, with and without the residual epilogue, and in place. The
sublayer is checked stage by stage through the intermediates it leaves in its
workspace, each stage against the oracle fed the previous GPU stage, plus the
whole chain against the float64 oracle end to end.
"""
import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W
from oracle import decode_ref as O
from tol import (FP32_ACC, FP32_ROT, check_float, check_float_sigma, check_kv_fp32,
                 check_ulp, rounded_operand_sigma)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def f64(t):
    return t.double().cpu().numpy()


# (B, N, K): Qwen3-0.6B-shaped QKV / O at batch 1, Llama-3-8B-shaped at batch 32, the
# serving mix at batch 256, and ragged batches for every batch tile.
SHAPES = [
    (1, 128, 64),
    (1, 4096, 1024),
    (1, 1024, 2048),
    (3, 384, 320),
    (17, 256, 512),
    (32, 6144, 4096),
    (32, 4096, 4096),
    (45, 640, 1152),
    (100, 512, 1024),
    (256, 3072, 2048),
    (300, 256, 256),
]


@pytest.mark.parametrize("B,N,K", SHAPES)
@pytest.mark.parametrize("with_residual", [True, False])
def test_linear(B, N, K, with_residual):
    inp = W.make_linear_inputs(B, N, K, seed=B * 7 + N + K, residual=with_residual)
    x, w = inp["x"].to(DEV), inp["w"].to(DEV)
    r = inp["residual"].to(DEV) if with_residual else None
    y = dsa.linear(x, w, r)
    torch.cuda.synchronize()
    ref = O.linear(f64(inp["x"]), f64(inp["w"]), f64(inp["residual"]) if with_residual else None)
    check_float(f64(y), ref, f"linear {B}x{N}x{K}")


NORM_SHAPES = [(1, 128, 64), (1, 4096, 1024), (3, 384, 320), (17, 256, 512), (32, 6144, 4096),
               (45, 640, 1152), (100, 512, 1024), (256, 3072, 2048), (300, 256, 256)]


def _norm_ref(inp, eps, with_residual=True):
    """The oracle's RMSNorm (unrounded) then its projection, h, and the spread the
    prologue's operand rounding gives each output (tol.rounded_operand_sigma)."""
    r = f64(inp["residual"]) if with_residual else None
    y_ref, h_ref = O.rmsnorm_residual(f64(inp["x"]), r, f64(inp["norm_w"]), eps)
    return O.linear(y_ref, f64(inp["w"])), h_ref, rounded_operand_sigma(y_ref, f64(inp["w"]))


@pytest.mark.parametrize("B,N,K", NORM_SHAPES)
@pytest.mark.parametrize("with_residual", [True, False])
def test_norm_linear(B, N, K, with_residual):
    """RMSNorm(x + residual) w^T with the norm as the projection's prologue, against the
    oracle's RMSNorm (unrounded) followed by its projection; h_out is x + residual."""
    eps = 1e-6
    inp = W.make_norm_linear_inputs(B, N, K, seed=B + 3 * N + K, residual=with_residual)
    x, w, nw = inp["x"].to(DEV), inp["w"].to(DEV), inp["norm_w"].to(DEV)
    r = inp["residual"].to(DEV) if with_residual else None
    h = torch.full((B, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(4, dtype=torch.int32, device=DEV)
    y = dsa.norm_linear(x, w, nw, residual=r, h_out=h, eps=eps, error_word=err)
    torch.cuda.synchronize()
    ref, h_ref, sig = _norm_ref(inp, eps, with_residual)
    check_float_sigma(f64(y), ref, sig, f"norm_linear {B}x{N}x{K}")
    check_ulp(f64(h), h_ref, "h = x + residual", 0.5)
    assert int(err[0].item()) == 0


@pytest.mark.parametrize("B,N,K", [(1, 6144, 4096), (32, 1024, 2048), (100, 384, 1024),
                                   (256, 256, 512)])
@pytest.mark.parametrize("k_split", range(1, 9))
def test_norm_linear_forced_splits(B, N, K, k_split):
    """Every cluster size: the sums of squares of the K slices are added across the
    cluster, so the row scale is that of the whole row."""
    if k_split > K // 64:
        pytest.skip("more slices than 64-wide K pieces")
    eps = 1e-5
    inp = W.make_norm_linear_inputs(B, N, K, seed=11 * k_split + B)
    h = torch.empty(B, K, dtype=torch.bfloat16, device=DEV)
    y = dsa.norm_linear(inp["x"].to(DEV), inp["w"].to(DEV), inp["norm_w"].to(DEV),
                        residual=inp["residual"].to(DEV), h_out=h, eps=eps, k_split=k_split)
    torch.cuda.synchronize()
    ref, h_ref, sig = _norm_ref(inp, eps)
    check_float_sigma(f64(y), ref, sig, f"norm_linear split {k_split}")
    check_ulp(f64(h), h_ref, "h", 0.5)


def test_norm_linear_matches_unfused_pair():
    """The prologue against K1 then the plain projection on the GPU: both within the
    oracle's bound, and h bit-identical to K1's residual output."""
    B, N, K, eps = 40, 1024, 2048, 1e-6
    inp = W.make_norm_linear_inputs(B, N, K, seed=77)
    x, w, nw, r = (inp[k].to(DEV) for k in ("x", "w", "norm_w", "residual"))
    r1 = r.clone()
    y1 = dsa.rmsnorm_residual(x, nw, residual=r1, eps=eps)
    p1 = dsa.linear(y1, w)
    h = torch.empty_like(r)
    p2 = dsa.norm_linear(x, w, nw, residual=r, h_out=h, eps=eps)
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), r1.view(torch.int16))
    assert torch.equal(r.view(torch.int16), inp["residual"].to(DEV).view(torch.int16))
    ref, _, sig = _norm_ref(inp, eps)
    check_float_sigma(f64(p1), ref, sig, "unfused")
    check_float_sigma(f64(p2), ref, sig, "prologue")


def test_linear_plans_cover_every_split():
    """The shapes above exercise the unsplit kernel and K split over clusters of CTAs."""
    splits = {dsa.linear_plan(B, N, K)[1] for B, N, K in SHAPES}
    assert 1 in splits and len(splits - {1}) >= 2, splits


@pytest.mark.parametrize("B,N,K", [(1, 6144, 4096), (32, 1024, 2048), (100, 384, 1024),
                                   (256, 256, 1024)])
@pytest.mark.parametrize("k_split", range(1, 9))
def test_linear_forced_splits(B, N, K, k_split):
    """Every cluster size, against the oracle, with no wait giving up."""
    inp = W.make_linear_inputs(B, N, K, seed=k_split)
    x, w, r = inp["x"].to(DEV), inp["w"].to(DEV), inp["residual"].to(DEV)
    err = torch.zeros(4, dtype=torch.int32, device=DEV)
    y = dsa.linear(x, w, r, error_word=err, k_split=k_split)
    torch.cuda.synchronize()
    check_float(f64(y), O.linear(f64(inp["x"]), f64(inp["w"]), f64(inp["residual"])),
                f"k_split {k_split}")
    assert int(err[0].item()) == 0


@pytest.mark.parametrize("B,N,K", [(1, 4096, 1024), (32, 6144, 4096), (256, 3072, 2048)])
def test_linear_repeats_bit_identical(B, N, K):
    """Slices are added in a fixed order: repeated calls give the same bits, and no
    wait gave up."""
    inp = W.make_linear_inputs(B, N, K, seed=5)
    x, w, r = inp["x"].to(DEV), inp["w"].to(DEV), inp["residual"].to(DEV)
    err = torch.zeros(4, dtype=torch.int32, device=DEV)
    y1 = dsa.linear(x, w, r, error_word=err)
    y2 = dsa.linear(x, w, r, error_word=err)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    check_float(f64(y1), O.linear(f64(inp["x"]), f64(inp["w"]), f64(inp["residual"])), "repeat")
    assert int(err[0].item()) == 0


def test_linear_in_place_residual():
    B, N, K = 24, 512, 768
    inp = W.make_linear_inputs(B, N, K, seed=9)
    x, w = inp["x"].to(DEV), inp["w"].to(DEV)
    yr = inp["residual"].to(DEV).clone()
    dsa.linear(x, w, yr, out=yr)
    torch.cuda.synchronize()
    check_float(f64(yr), O.linear(f64(inp["x"]), f64(inp["w"]), f64(inp["residual"])), "in place")


def test_linear_special_values():
    """One-hot rows select weight columns exactly; a zero weight returns the residual
    bit for bit."""
    B, N, K = 64, 256, 192
    eye = torch.zeros(B, K, dtype=torch.bfloat16)
    for b in range(B):
        eye[b, (5 * b) % K] = 1.0
    w = W.make_linear_inputs(1, N, K, seed=3)["w"]
    y = dsa.linear(eye.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    for b in range(B):
        assert torch.equal(y[b].cpu(), w[:, (5 * b) % K])
    r = W.make_linear_inputs(B, N, K, seed=4)["residual"].to(DEV)
    z = dsa.linear(eye.to(DEV), torch.zeros(N, K, dtype=torch.bfloat16, device=DEV), r)
    torch.cuda.synchronize()
    assert torch.equal(z.view(torch.int16), r.view(torch.int16))


def test_linear_empty_batch():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(128, 256, dtype=torch.bfloat16, device=DEV)
    y = dsa.linear(x, w)
    assert y.shape == (0, 128)


# ------------------------------------------------------------ sublayer ---
SUB = {
    "tiny": W.TINY,
    "qwen3_ctx128": W.QWEN3_128,
    "llama3_small": W.small_variant(W.LLAMA3_BATCHED, B=6, max_len=900),
    "serving_small": W.small_variant(W.SERVING_MIX, B=40, max_len=700),
    "long_small": W.small_variant(W.LONG_CONTEXT, max_len=3000),
}


def _run_sublayer(cfg, window=0, with_residual=True, graph=False, inv_freq=None, scale=0.0):
    inp = W.make_inputs(cfg)
    wts = W.make_projection_weights(cfg)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    T_cap = inp["k_cache"].shape[2]
    nbytes = dsa.sublayer_workspace_bytes(B, H, Hq, Hkv, D, T_cap)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(B, H, dtype=torch.bfloat16, device=DEV)
    res = d["residual"].clone() if with_residual else None
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    kw = dict(x=d["x"], residual=res, norm_w=d["norm_w"], w_qkv=wts["w_qkv"].to(DEV),
              w_o=wts["w_o"].to(DEV), k_cache=kc, v_cache=vc, pos=d["pos"], lens=d["lens"],
              out=out, workspace=ws, theta=cfg.theta, layout=cfg.layout,
              q_norm_w=d.get("q_norm_w"), k_norm_w=d.get("k_norm_w"), eps=cfg.eps,
              window=window, inv_freq=inv_freq, scale=scale)
    if graph:
        g = dsa.StepGraph(step=dsa.attn_sublayer, **kw)
        # the eager warm-up inside StepGraph already ran one step: restore the inputs
        if res is not None:
            res.copy_(d["residual"])
        kc.copy_(d["k_cache"])
        vc.copy_(d["v_cache"])
        g.replay()
    else:
        dsa.attn_sublayer(**kw)
    torch.cuda.synchronize()
    views = dsa.sublayer_views(ws, B, H, Hq, Hkv, D, T_cap)
    return inp, wts, {"out": out, "h": res, "k_cache": kc, "v_cache": vc, "ws": ws, **views}


def _check_stages(cfg, inp, wts, g, window=0, with_residual=True, ref_freq=None, scale=None):
    B, Hq, Hkv, D = cfg.B, cfg.Hq, cfg.Hkv, cfg.D
    x = f64(inp["x"])
    r = f64(inp["residual"]) if with_residual else None
    y_ref, h_ref = O.rmsnorm_residual(x, r, f64(inp["norm_w"]), cfg.eps)
    if with_residual:
        check_ulp(f64(g["h"]), h_ref, "h = x + residual", 0.5)
    check_float(f64(g["y"]), y_ref, "RMSNorm")
    qkv_ref = O.linear(f64(g["y"]), f64(wts["w_qkv"]))
    if D == 128:
        # the projection's epilogue rotates and appends; the packed qkv is not stored
        q, k_new, v_new = O.split_qkv(qkv_ref, Hq, Hkv, D)
    else:
        check_float(f64(g["qkv"]), qkv_ref, "QKV projection")
        q, k_new, v_new = O.split_qkv(f64(g["qkv"]), Hq, Hkv, D)
    qn = f64(inp["q_norm_w"]) if cfg.qk_norm else None
    kn = f64(inp["k_norm_w"]) if cfg.qk_norm else None
    q_ref, kc_ref, vc_ref = O.qknorm_rope_kv_append(q, k_new, v_new, qn, kn, f64(inp["k_cache"]),
                                                    f64(inp["v_cache"]), inp["pos"].numpy(),
                                                    cfg.theta, cfg.layout, cfg.eps, ref_freq)
    check_float(f64(g["q_rot"]), q_ref, "rotated q")
    pos = inp["pos"].numpy()
    kc, vc = f64(g["k_cache"]), f64(g["v_cache"])
    if D == 128:  # straight from the fp32 projection (its epilogue rotates)
        ek, ev = _kv_fp32_bounds(f64(g["y"]), f64(wts["w_qkv"]), cfg, kn)
    for b in range(B):
        if D == 128:
            check_kv_fp32(kc[b, :, pos[b]], kc_ref[b, :, pos[b]], ek[b], "appended K")
            check_kv_fp32(vc[b, :, pos[b]], vc_ref[b, :, pos[b]], ev[b], "appended V")
        else:
            check_ulp(kc[b, :, pos[b]], kc_ref[b, :, pos[b]], "appended K", 1.0)
            assert np.array_equal(vc[b, :, pos[b]], vc_ref[b, :, pos[b]]), "appended V"
    attn_ref = O.gqa_decode_attention(f64(g["q_rot"]), kc, vc, inp["lens"].numpy(), scale,
                                      window=window or None)
    check_float(f64(g["attn"]), attn_ref, "attention")
    h_gpu = f64(g["h"]) if with_residual else x
    out_ref = O.linear(f64(g["attn"]).reshape(B, Hq * D), f64(wts["w_o"]), h_gpu)
    check_float(f64(g["out"]), out_ref, "output projection + residual")
    assert dsa.device_errors(g["ws"]) == 0


@pytest.mark.parametrize("name", list(SUB))
def test_sublayer_stages(name):
    cfg = SUB[name]
    inp, wts, g = _run_sublayer(cfg)
    _check_stages(cfg, inp, wts, g)


def test_sublayer_without_residual_and_windowed():
    cfg = SUB["serving_small"]
    inp, wts, g = _run_sublayer(cfg, window=256, with_residual=False)
    _check_stages(cfg, inp, wts, g, window=256, with_residual=False)


@pytest.mark.parametrize("name", ["qwen3_ctx128", "llama3_small"])
def test_sublayer_end_to_end(name):
    """The whole chain against the float64 oracle with no GPU intermediates. Every
    stage rounds to bf16 once (relative error 2^-9 each): h and out at the scale of
    out, and y, qkv, the rotated q / K, the attention rows at the scale of the
    projected part a W_o^T, so ||out - ref|| <= 2 * 2^-9 ||ref|| + 5 * 2^-9 ||a W_o^T||."""
    cfg = SUB[name]
    inp, wts, g = _run_sublayer(cfg)
    f = {k: (f64(v) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    f.update(eps=cfg.eps, theta=cfg.theta, layout=cfg.layout, Hq=cfg.Hq, Hkv=cfg.Hkv, D=cfg.D,
             w_qkv=f64(wts["w_qkv"]), w_o=f64(wts["w_o"]), pos=inp["pos"].numpy(),
             lens=inp["lens"].numpy())
    if not cfg.qk_norm:
        f["q_norm_w"] = f["k_norm_w"] = None
    ref = O.attention_sublayer(f)
    gpu = f64(g["out"])
    u = 2.0 ** -9
    err = np.linalg.norm(gpu - ref["out"])
    bound = 2 * u * np.linalg.norm(ref["out"]) + 5 * u * np.linalg.norm(ref["out"] - ref["h"])
    assert err <= bound, (err, bound)


@pytest.mark.parametrize("name", ["tiny", "llama3_small", "serving_small"])
def test_sublayer_rope_table(name):
    """The sublayer with an NTK-aware table (head_dim 64: the rotation launch; 128: the
    projection's epilogue), each stage against the oracle with its own table."""
    cfg = SUB[name]
    factor = 4.0
    inp, wts, g = _run_sublayer(cfg, inv_freq=dsa.rope_inv_freq(cfg.D, cfg.theta, "ntk", factor))
    _check_stages(cfg, inp, wts, g,
                  ref_freq=O.rope_scaled_inv_freq(cfg.D, np.float32(cfg.theta), "ntk", factor))


@pytest.mark.parametrize("name", ["tiny", "qwen3_ctx128", "llama3_small"])
def test_sublayer_yarn(name):
    """The sublayer with a YaRN table and its softmax scale; the attention stage against
    the oracle's form of the method (rotated q and K both times 0.1 ln(s) + 1 under
    the plain 1/sqrt(D) scale), the other stages against the oracle with its own table."""
    cfg = SUB[name]
    s, ctx = 8.0, 128
    inp, wts, g = _run_sublayer(cfg, inv_freq=dsa.rope_inv_freq(cfg.D, cfg.theta, "yarn", s, ctx),
                                scale=dsa.yarn_softmax_scale(cfg.D, s))
    m = O.yarn_attention_factor(s)
    _check_stages(cfg, inp, wts, g,
                  ref_freq=O.rope_scaled_inv_freq(cfg.D, np.float32(cfg.theta), "yarn", s, ctx),
                  scale=m * m / np.sqrt(cfg.D))


@pytest.mark.parametrize("name", ["qwen3_ctx128", "serving_small"])
def test_norm_qkv_projection_rope_table(name):
    """The RMSNorm-prologue QKV projection with a linear-interpolation table against
    the unfused pair (RMSNorm, then the projection with the rotation epilogue) given
    the same table, and the rotated q against the oracle with its own table."""
    cfg = SUB[name]
    inp = W.make_inputs(cfg)
    wts = W.make_projection_weights(cfg)
    factor = 8.0
    t = dsa.rope_inv_freq(cfg.D, cfg.theta, "linear", factor)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    qn = d["q_norm_w"] if cfg.qk_norm else None
    kn = d["k_norm_w"] if cfg.qk_norm else None
    kc1, vc1 = d["k_cache"].clone(), d["v_cache"].clone()
    q1 = dsa.norm_qkv_proj_rope_append(d["x"], wts["w_qkv"].to(DEV), d["norm_w"], kc1, vc1,
                                       d["pos"], cfg.theta, cfg.layout, residual=d["residual"],
                                       q_norm_w=qn, k_norm_w=kn, eps=cfg.eps, inv_freq=t)
    y = dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=d["residual"].clone(), eps=cfg.eps)
    kc2, vc2 = d["k_cache"].clone(), d["v_cache"].clone()
    q2 = dsa.qkv_proj_rope_append(y, wts["w_qkv"].to(DEV), kc2, vc2, d["pos"], cfg.theta,
                                  cfg.layout, qn, kn, cfg.eps, inv_freq=t)
    torch.cuda.synchronize()
    y_ref, _ = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]),
                                  cfg.eps)
    qs, ks, vs = O.split_qkv(O.linear(y_ref, f64(wts["w_qkv"])), cfg.Hq, cfg.Hkv, cfg.D)
    ref_t = O.rope_scaled_inv_freq(cfg.D, np.float32(cfg.theta), "linear", factor)
    q_ref, _, _ = O.qknorm_rope_kv_append(
        qs, ks, vs, f64(inp["q_norm_w"]) if cfg.qk_norm else None,
        f64(inp["k_norm_w"]) if cfg.qk_norm else None, f64(inp["k_cache"]), f64(inp["v_cache"]),
        inp["pos"].numpy(), cfg.theta, cfg.layout, cfg.eps, ref_t)
    sq, _, _ = O.split_qkv(rounded_operand_sigma(y_ref, f64(wts["w_qkv"])), cfg.Hq, cfg.Hkv,
                           cfg.D)
    sq = _rotated_sigma(sq, qs, f64(inp["q_norm_w"]) if cfg.qk_norm else None, cfg)
    check_float_sigma(f64(q1), q_ref, sq, "fused rotated q")
    check_float_sigma(f64(q2), q_ref, sq, "unfused rotated q")


def test_sublayer_graph_replay_matches_eager():
    cfg = SUB["llama3_small"]
    _, _, eager = _run_sublayer(cfg)
    _, _, graphed = _run_sublayer(cfg, graph=True)
    assert torch.equal(eager["out"].view(torch.int16), graphed["out"].view(torch.int16))
    assert torch.equal(eager["k_cache"].view(torch.int16), graphed["k_cache"].view(torch.int16))


@pytest.mark.parametrize("name", ["qwen3_ctx128", "llama3_small", "serving_small", "long_small"])
@pytest.mark.parametrize("with_residual", [True, False])
def test_norm_qkv_projection_with_rotation(name, with_residual):
    """The packed QKV projection with the RMSNorm prologue and the rotation epilogue,
    against the oracle's RMSNorm, projection and rotation step in float64."""
    cfg = SUB[name]
    inp = W.make_inputs(cfg)
    wts = W.make_projection_weights(cfg)
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    err = torch.zeros(4, dtype=torch.int32, device=DEV)
    qn = inp["q_norm_w"].to(DEV) if cfg.qk_norm else None
    kn = inp["k_norm_w"].to(DEV) if cfg.qk_norm else None
    r = inp["residual"].to(DEV) if with_residual else None
    h = torch.empty(B, H, dtype=torch.bfloat16, device=DEV) if with_residual else None
    q = dsa.norm_qkv_proj_rope_append(inp["x"].to(DEV), wts["w_qkv"].to(DEV),
                                      inp["norm_w"].to(DEV), kc, vc, inp["pos"].to(DEV),
                                      cfg.theta, cfg.layout, residual=r, h_out=h, q_norm_w=qn,
                                      k_norm_w=kn, eps=cfg.eps, error_word=err)
    torch.cuda.synchronize()
    y_ref, h_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]) if with_residual
                                      else None, f64(inp["norm_w"]), cfg.eps)
    if with_residual:
        check_ulp(f64(h), h_ref, "h", 0.5)
    qs, ks, vs = O.split_qkv(O.linear(y_ref, f64(wts["w_qkv"])), Hq, Hkv, D)
    q_ref, kc_ref, vc_ref = O.qknorm_rope_kv_append(
        qs, ks, vs, f64(inp["q_norm_w"]) if cfg.qk_norm else None,
        f64(inp["k_norm_w"]) if cfg.qk_norm else None, f64(inp["k_cache"]), f64(inp["v_cache"]),
        inp["pos"].numpy(), cfg.theta, cfg.layout, cfg.eps)
    sq, sk, sv = O.split_qkv(rounded_operand_sigma(y_ref, f64(wts["w_qkv"])), Hq, Hkv, D)
    sq = _rotated_sigma(sq, qs, f64(inp["q_norm_w"]) if cfg.qk_norm else None, cfg)
    sk = _rotated_sigma(sk, ks, f64(inp["k_norm_w"]) if cfg.qk_norm else None, cfg)
    check_float_sigma(f64(q), q_ref, sq, "rotated q")
    pos = inp["pos"].numpy()
    kg, vg = f64(kc), f64(vc)
    for b in range(B):
        check_float_sigma(kg[b, :, pos[b]], kc_ref[b, :, pos[b]], sk[b], "appended K")
        check_float_sigma(vg[b, :, pos[b]], vc_ref[b, :, pos[b]], sv[b], "appended V")
    assert int(err[0].item()) == 0
    # stage-wise: the oracle's projection and rotation fed the operand the prologue forms
    # (u = bf16((x + r) * w), fp32 sum and product as in the kernel) and the row scale
    # rsqrt(mean((x + r)^2) + eps); the KV-cache writes then sit within one bf16 ulp
    u, rs = _prologue_operand(inp["x"], inp["residual"] if with_residual else None,
                              inp["norm_w"], cfg.eps)
    qs_u, ks_u, vs_u = O.split_qkv(rs * O.linear(u, f64(wts["w_qkv"])), Hq, Hkv, D)
    q_u, kc_u, vc_u = O.qknorm_rope_kv_append(
        qs_u, ks_u, vs_u, f64(inp["q_norm_w"]) if cfg.qk_norm else None,
        f64(inp["k_norm_w"]) if cfg.qk_norm else None, f64(inp["k_cache"]), f64(inp["v_cache"]),
        pos, cfg.theta, cfg.layout, cfg.eps)
    check_float(f64(q), q_u, "rotated q, stage-wise")
    ek, ev = _kv_fp32_bounds(u, f64(wts["w_qkv"]), cfg,
                             f64(inp["k_norm_w"]) if cfg.qk_norm else None, rs)
    for b in range(B):
        check_kv_fp32(kg[b, :, pos[b]], kc_u[b, :, pos[b]], ek[b], "appended K, stage-wise")
        check_kv_fp32(vg[b, :, pos[b]], vc_u[b, :, pos[b]], ev[b], "appended V, stage-wise")


def _prologue_operand(x, residual, norm_w, eps):
    """The RMSNorm prologue's tensor-core operand and row scale, in the precision the
    projection forms them: s = x + r and s * w in fp32, rounded to bf16 once (round to
    nearest even); the row scale from the exact s in fp64."""
    x32 = x.float().numpy()
    s32 = x32 + residual.float().numpy() if residual is not None else x32
    u = torch.from_numpy(s32 * norm_w.float().numpy()[None, :]).to(torch.bfloat16)
    s64 = f64(x) + (f64(residual) if residual is not None else 0.0)
    rs = 1.0 / np.sqrt(np.mean(s64 * s64, axis=1, keepdims=True) + eps)
    return f64(u), rs


def _kv_fp32_bounds(u, w_qkv, cfg, k_norm_w=None, row_scale=None):
    """The fp32 error bounds E of the K and V slot writes of a QKV projection whose
    rotation runs in its epilogue (tests/tol.py): V carries its accumulation bound, K the
    accumulation bounds of the element and its pair partner through the QK-norm, plus
    the rotation's own. u: the operand [B, hidden] (fp64); k_norm_w: [D] or None;
    row_scale: the RMSNorm prologue's per-row scale [B, 1] or None. Returns (E_k, E_v),
    each [B, Hkv, D]."""
    S = np.abs(u) @ np.abs(w_qkv).T  # sum_k |u_k W_nk| per (row, feature)
    acc = u @ w_qkv.T
    if row_scale is not None:
        S, acc = S * row_scale, acc * row_scale
    _, sk, sv = O.split_qkv(FP32_ACC * S, cfg.Hq, cfg.Hkv, cfg.D)
    _, ks, _ = O.split_qkv(acc, cfg.Hq, cfg.Hkv, cfg.D)
    if k_norm_w is not None:  # the norm scales each element by rstd * w
        rstd = 1.0 / np.sqrt(np.mean(ks * ks, axis=-1, keepdims=True) + cfg.eps)
        sk = sk * rstd * np.abs(k_norm_w)
        ks = ks * rstd * np.abs(k_norm_w)
    d = np.arange(cfg.D)
    partner = (d + cfg.D // 2) % cfg.D if cfg.layout == "neox" else d ^ 1
    ek = sk + sk[..., partner] + FP32_ROT * (np.abs(ks) + np.abs(ks[..., partner]))
    return ek, sv


def _rotated_sigma(sig, heads, norm_w, cfg):
    """The spread of a projected head's features carried through the rotation step:
    the QK-norm scales feature d by rsqrt(mean square + eps) * |w_d|, the rotation mixes
    d with its partner (NeoX d + D/2, interleaved d ^ 1) by cos / sin, so the spreads add
    in quadrature."""
    D = sig.shape[-1]
    if norm_w is not None:
        rstd = 1.0 / np.sqrt(np.mean(heads * heads, axis=-1, keepdims=True) + cfg.eps)
        sig = sig * rstd * np.abs(norm_w)
    d = np.arange(D)
    partner = (d + D // 2) % D if cfg.layout == "neox" else d ^ 1
    return np.sqrt(sig * sig + sig[..., partner] ** 2)


@pytest.mark.parametrize("name", ["qwen3_ctx128", "llama3_small", "serving_small", "long_small"])
def test_qkv_projection_with_rotation(name):
    """The packed QKV projection whose epilogue is QK-norm + RoPE + the K/V append,
    against the oracle's projection (unrounded) followed by the rotation step; every
    other cache slot is left bit for bit."""
    cfg = SUB[name]
    inp = W.make_inputs(cfg)
    wts = W.make_projection_weights(cfg)
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    y = W.make_linear_inputs(B, 8, H, seed=3)["x"]  # a normalised-looking input row block
    kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    err = torch.zeros(4, dtype=torch.int32, device=DEV)
    qn = inp["q_norm_w"].to(DEV) if cfg.qk_norm else None
    kn = inp["k_norm_w"].to(DEV) if cfg.qk_norm else None
    q = dsa.qkv_proj_rope_append(y.to(DEV), wts["w_qkv"].to(DEV), kc, vc, inp["pos"].to(DEV),
                                 cfg.theta, cfg.layout, qn, kn, cfg.eps, error_word=err)
    torch.cuda.synchronize()
    qkv = O.linear(f64(y), f64(wts["w_qkv"]))
    qs, ks, vs = O.split_qkv(qkv, Hq, Hkv, D)
    q_ref, kc_ref, vc_ref = O.qknorm_rope_kv_append(
        qs, ks, vs, f64(inp["q_norm_w"]) if cfg.qk_norm else None,
        f64(inp["k_norm_w"]) if cfg.qk_norm else None, f64(inp["k_cache"]), f64(inp["v_cache"]),
        inp["pos"].numpy(), cfg.theta, cfg.layout, cfg.eps)
    check_float(f64(q), q_ref, "rotated q")
    pos = inp["pos"].numpy()
    kg, vg = f64(kc), f64(vc)
    # the KV-cache writes: within one bf16 ulp of the exact result, or of the fp32
    # accumulation's error where the result is tiny against its terms
    ek, ev = _kv_fp32_bounds(f64(y), f64(wts["w_qkv"]), cfg,
                             f64(inp["k_norm_w"]) if cfg.qk_norm else None)
    for b in range(B):
        check_kv_fp32(kg[b, :, pos[b]], kc_ref[b, :, pos[b]], ek[b], "appended K")
        check_kv_fp32(vg[b, :, pos[b]], vc_ref[b, :, pos[b]], ev[b], "appended V")
    mask = np.ones(kg.shape[:3], dtype=bool)
    for b in range(B):
        mask[b, :, pos[b]] = False
    k0 = inp["k_cache"].view(torch.int16).numpy()
    v0 = inp["v_cache"].view(torch.int16).numpy()
    assert np.array_equal(kc.view(torch.int16).cpu().numpy()[mask], k0[mask])
    assert np.array_equal(vc.view(torch.int16).cpu().numpy()[mask], v0[mask])
    assert int(err[0].item()) == 0
