"""The kernels reading and writing pinned host memory directly (GPU only).

Arguments documented as [device|host] may be page-locked, mapped host memory: the
kernels then cross the host link themselves and a host-to-host decode step needs no
copy step. The same kernels run on the same values either way, so every result here
must be bit-identical to the device-resident call's, and a pointer the kernels could
not reach must be refused before anything launches.
"""
import ctypes

import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
CONFIGS = {
    "tiny": W.TINY,
    "qwen3_ctx128": W.QWEN3_128,
    "serving_small": W.small_variant(W.SERVING_MIX, B=40, max_len=700),
}


def same(a, b, what):
    a, b = a.detach().cpu(), b.detach().cpu()
    assert a.shape == b.shape and a.dtype == b.dtype, what
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), what


def pinned(t):
    return t.detach().cpu().clone().pin_memory()


def on_dev(t):
    return None if t is None else t.to(DEV)


def device_step(cfg, inp, window=0, whole=False, **rope):
    """The device-resident reference for the host-staged forms: K1, K2 and the attention
    as separate calls (the kernels the host-staged step uses), or (whole) decode_step,
    which short contexts run as one kernel."""
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    max_len = int(inp["lens"].max())
    B, Hq, D = d["q"].shape
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    r = {"y": torch.empty_like(d["x"]), "residual": d["residual"].clone(), "q": d["q"].clone(),
         "k_cache": d["k_cache"].clone(), "v_cache": d["v_cache"].clone(),
         "out": torch.empty_like(d["q"])}
    if whole:
        dsa.decode_step(d["x"], r["residual"], d["norm_w"], r["y"], r["q"], d["k_new"],
                        d["v_new"], r["k_cache"], r["v_cache"], d["pos"], d["lens"], r["out"], ws,
                        theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                        k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len, window=window,
                        **rope)
    else:
        dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=r["residual"], eps=cfg.eps,
                             out=r["y"])
        dsa.qknorm_rope_kv_append(r["q"], d["k_new"], d["v_new"], r["k_cache"], r["v_cache"],
                                  d["pos"], cfg.theta, cfg.layout, d["q_norm_w"], d["k_norm_w"],
                                  cfg.eps)
        dsa.gqa_decode_attn(r["q"], r["k_cache"], r["v_cache"], d["lens"], max_len=max_len,
                            workspace=ws, out=r["out"], window=window)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    return r


class HostStep:
    """A host-to-host decode step: inputs and results in pinned host memory, caches,
    weights, the rotated q and the workspace on the device. K2 reads its inputs from
    the host; K1 runs on a second stream forked after K2, beside the attention."""

    def __init__(self, cfg, inp, window=0):
        self.cfg, self.window = cfg, window
        self.h = {k: pinned(inp[k]) for k in ("x", "residual", "q", "k_new", "v_new", "pos",
                                              "lens")}
        self.h["y"] = torch.empty(tuple(inp["x"].shape), dtype=torch.bfloat16, pin_memory=True)
        self.h["out"] = torch.empty(tuple(inp["q"].shape), dtype=torch.bfloat16, pin_memory=True)
        self.d = {k: on_dev(inp[k]) for k in ("k_cache", "v_cache", "norm_w", "q_norm_w",
                                              "k_norm_w")}
        self.q = torch.empty(tuple(inp["q"].shape), dtype=torch.bfloat16, device=DEV)
        self.max_len = int(inp["lens"].max())
        B, Hq, D = inp["q"].shape
        self.ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, self.max_len)
        self.side = torch.cuda.Stream()

    def k2(self):
        c, h, d = self.cfg, self.h, self.d
        dsa.qknorm_rope_kv_append(h["q"], h["k_new"], h["v_new"], d["k_cache"], d["v_cache"],
                                  h["pos"], c.theta, c.layout, d["q_norm_w"], d["k_norm_w"],
                                  c.eps, q_out=self.q)

    def attn(self):
        dsa.gqa_decode_attn(self.q, self.d["k_cache"], self.d["v_cache"], self.h["lens"],
                            max_len=self.max_len, workspace=self.ws, out=self.h["out"],
                            window=self.window)

    def k1(self):
        dsa.rmsnorm_residual(self.h["x"], self.d["norm_w"], residual=self.h["residual"],
                             eps=self.cfg.eps, out=self.h["y"])

    def eager(self):
        main = torch.cuda.current_stream()
        self.k2()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            self.k1()
        self.attn()
        main.wait_stream(self.side)


def check_against(r, hs, inp):
    same(hs.h["y"], r["y"], "y")
    same(hs.h["residual"], r["residual"], "residual")
    same(hs.q, r["q"], "rotated q")
    same(hs.h["out"], r["out"], "out")
    same(hs.d["k_cache"], r["k_cache"], "k_cache")
    same(hs.d["v_cache"], r["v_cache"], "v_cache")
    same(hs.h["q"], inp["q"], "q_in untouched")
    assert dsa.device_errors(hs.ws) == 0


@pytest.mark.parametrize("name", list(CONFIGS))
@pytest.mark.parametrize("window", [0, 33])
def test_zero_copy_step_matches_device_step(name, window):
    cfg = CONFIGS[name]
    inp = W.make_inputs(cfg)
    r = device_step(cfg, inp, window)
    hs = HostStep(cfg, inp, window)
    hs.eager()
    torch.cuda.synchronize()
    check_against(r, hs, inp)


def test_zero_copy_step_graph_replays():
    """The same schedule captured in a StepGraph (K2 as the prologue, K1 as a branch);
    two replays with the host inputs restored in between give the device result."""
    cfg = CONFIGS["serving_small"]
    inp = W.make_inputs(cfg)
    r = device_step(cfg, inp)
    hs = HostStep(cfg, inp)
    g = dsa.StepGraph(prologue=hs.k2, step=hs.attn, branches=[dsa.GraphBranch(hs.k1)])
    for _ in range(2):
        hs.h["residual"].copy_(inp["residual"])  # K1 updates it in place
        hs.h["y"].zero_()
        hs.h["out"].zero_()
        g.replay()
        torch.cuda.synchronize()
        check_against(r, hs, inp)


@pytest.mark.parametrize("name", ["qwen3_ctx128", "serving_small"])  # one and three launches
def test_decode_step_with_host_arguments(name):
    """The whole-step call itself with every [device|host] argument but q in pinned host
    memory, on the one-launch path and on the three-launch path."""
    cfg = CONFIGS[name]
    inp = W.make_inputs(cfg)
    r = device_step(cfg, inp, whole=True)
    h = {k: pinned(inp[k]) for k in ("x", "residual", "k_new", "v_new", "pos", "lens")}
    y = torch.empty(tuple(inp["x"].shape), dtype=torch.bfloat16, pin_memory=True)
    out = torch.empty(tuple(inp["q"].shape), dtype=torch.bfloat16, pin_memory=True)
    q = inp["q"].to(DEV)
    kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    max_len = int(inp["lens"].max())
    B, Hq, D = q.shape
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    dsa.decode_step(h["x"], h["residual"], inp["norm_w"].to(DEV), y, q, h["k_new"], h["v_new"],
                    kc, vc, h["pos"], h["lens"], out, ws, theta=cfg.theta, layout=cfg.layout,
                    q_norm_w=on_dev(inp["q_norm_w"]), k_norm_w=on_dev(inp["k_norm_w"]),
                    eps=cfg.eps, max_len=max_len)
    torch.cuda.synchronize()
    for k, v in (("y", y), ("residual", h["residual"]), ("q", q), ("out", out), ("k_cache", kc),
                 ("v_cache", vc)):
        same(v, r[k], k)


@pytest.mark.parametrize("name", ["qwen3_ctx128", "serving_small"])  # one and three launches
def test_decode_step_host_arguments_with_yarn(name):
    """A YaRN frequency table and its softmax scale on the host-staged whole step: the
    same bits as the device-resident call given the same table and scale."""
    cfg = CONFIGS[name]
    inp = W.make_inputs(cfg)
    rope = dict(inv_freq=dsa.rope_inv_freq(cfg.D, cfg.theta, "yarn", 4.0, 64),
                scale=dsa.yarn_softmax_scale(cfg.D, 4.0))
    r = device_step(cfg, inp, whole=True, **rope)
    h = {k: pinned(inp[k]) for k in ("x", "residual", "k_new", "v_new", "pos", "lens")}
    y = torch.empty(tuple(inp["x"].shape), dtype=torch.bfloat16, pin_memory=True)
    out = torch.empty(tuple(inp["q"].shape), dtype=torch.bfloat16, pin_memory=True)
    q = inp["q"].to(DEV)
    kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    max_len = int(inp["lens"].max())
    B, Hq, D = q.shape
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    dsa.decode_step(h["x"], h["residual"], inp["norm_w"].to(DEV), y, q, h["k_new"], h["v_new"],
                    kc, vc, h["pos"], h["lens"], out, ws, theta=cfg.theta, layout=cfg.layout,
                    q_norm_w=on_dev(inp["q_norm_w"]), k_norm_w=on_dev(inp["k_norm_w"]),
                    eps=cfg.eps, max_len=max_len, **rope)
    torch.cuda.synchronize()
    for k, v in (("y", y), ("residual", h["residual"]), ("q", q), ("out", out), ("k_cache", kc),
                 ("v_cache", vc)):
        same(v, r[k], k)


def test_k2_into_q_out_matches_in_place():
    cfg = CONFIGS["serving_small"]
    inp = W.make_inputs(cfg)
    args = dict(theta=cfg.theta, layout=cfg.layout, q_norm_w=on_dev(inp["q_norm_w"]),
                k_norm_w=on_dev(inp["k_norm_w"]), eps=cfg.eps)
    q1 = inp["q"].to(DEV)
    kc1, vc1 = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    dsa.qknorm_rope_kv_append(q1, inp["k_new"].to(DEV), inp["v_new"].to(DEV), kc1, vc1,
                              inp["pos"].to(DEV), **args)
    q_in = inp["q"].to(DEV)
    q2 = torch.full_like(q_in, float("nan"))
    kc2, vc2 = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    dsa.qknorm_rope_kv_append(q_in, inp["k_new"].to(DEV), inp["v_new"].to(DEV), kc2, vc2,
                              inp["pos"].to(DEV), q_out=q2, **args)
    torch.cuda.synchronize()
    same(q2, q1, "q_out")
    same(q_in, inp["q"], "q_in untouched")
    same(kc2, kc1, "k_cache")
    same(vc2, vc1, "v_cache")


def test_linear_with_host_residual_and_out():
    lin = W.make_linear_inputs(24, 512, 256, seed=5)
    x, w = lin["x"].to(DEV), lin["w"].to(DEV)
    ref = dsa.linear(x, w, lin["residual"].to(DEV))
    res_h = pinned(lin["residual"])
    out_h = torch.empty((24, 512), dtype=torch.bfloat16, pin_memory=True)
    dsa.linear(x, w, res_h, out=out_h)
    torch.cuda.synchronize()
    same(out_h, ref, "y")


@pytest.mark.parametrize("temperature", [0.0, 0.8])
def test_sampler_with_host_rows(temperature):
    smp = W.make_sampler_inputs(6, 5000, "peaked", L=12, seed=9)
    u = torch.rand(6, generator=torch.Generator().manual_seed(3))
    kw = dict(penalty=1.2, temperature=temperature, top_p=0.9, top_k=50)
    ref = dsa.sample(smp["logits"].to(DEV), smp["ids"].to(DEV), u=u.to(DEV), **kw)
    got = dsa.sample(pinned(smp["logits"]), pinned(smp["ids"]), u=pinned(u), **kw)
    torch.cuda.synchronize()
    assert not got.is_cuda
    same(got, ref, "tokens")


def test_unreachable_pointers_are_refused():
    """Pageable host memory anywhere, or pinned host memory where the kernels use bulk
    copies, is refused on the host with DEC_ERR_INVALID_ARG and nothing launches."""
    L = dsa.lib()
    B, hidden = 4, 256
    raw = np.zeros(B * hidden + 64, dtype=np.uint16)  # pageable; 16-byte aligned view
    skip = (-raw.ctypes.data % 16) // 2
    x_pageable = raw[skip:skip + B * hidden]
    w = torch.ones(hidden, dtype=torch.bfloat16, device=DEV)
    y = torch.full((B, hidden), 7.0, dtype=torch.bfloat16, device=DEV)
    st = L.dec_rmsnorm_residual(ctypes.c_void_p(x_pageable.ctypes.data), None, dsa._ptr(w),
                                dsa._ptr(y), B, hidden, 1e-6, dsa._stream(None))
    assert st == 1 and b"neither device memory" in L.dec_last_error()
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()), "a refused call must launch nothing"

    cfg = W.TINY
    inp = W.make_inputs(cfg)
    max_len = int(inp["lens"].max())
    B, Hq, D = inp["q"].shape
    T_cap = inp["k_cache"].shape[2]
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    q, vc, lens = inp["q"].to(DEV), inp["v_cache"].to(DEV), inp["lens"].to(DEV)
    kc_host = pinned(inp["k_cache"])
    out = torch.full_like(q, 7.0)
    st = L.dec_gqa_decode_attn(dsa._ptr(q), dsa._ptr(kc_host), dsa._ptr(vc), dsa._ptr(lens),
                               dsa._ptr(out), B, Hq, cfg.Hkv, D, T_cap, max_len, 0.0, 0,
                               dsa._ptr(ws), ws.numel(), dsa._stream(None))
    assert st == 1 and b"k_cache must be device memory" in L.dec_last_error()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a refused call must launch nothing"
    with pytest.raises(ValueError, match="pinned host tensor"):
        dsa.rmsnorm_residual(inp["x"], inp["norm_w"].to(DEV))  # pageable CPU tensor


def test_one_launch_step_host_to_host():
    """Short contexts run as one kernel, whose q is read and written with plain loads
    and stores: with q and every other [device|host] argument in pinned host memory the
    step gives the device step's results bit for bit. The three-launch path keeps q on
    the device (its split pass reads q with bulk copies) and refuses a host q."""
    cfg = CONFIGS["qwen3_ctx128"]
    inp = W.make_inputs(cfg)
    B, Hq, D = inp["q"].shape
    max_len = int(inp["lens"].max())
    assert dsa.decode_step_launches(B, Hq, cfg.Hkv, D, max_len) == 1
    r = device_step(cfg, inp, whole=True)
    h = {k: pinned(inp[k]) for k in ("x", "residual", "q", "k_new", "v_new", "pos", "lens")}
    y = torch.empty(tuple(inp["x"].shape), dtype=torch.bfloat16, pin_memory=True)
    out = torch.empty(tuple(inp["q"].shape), dtype=torch.bfloat16, pin_memory=True)
    kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    dsa.decode_step(h["x"], h["residual"], inp["norm_w"].to(DEV), y, h["q"], h["k_new"],
                    h["v_new"], kc, vc, h["pos"], h["lens"], out, ws, theta=cfg.theta,
                    layout=cfg.layout, q_norm_w=on_dev(inp["q_norm_w"]),
                    k_norm_w=on_dev(inp["k_norm_w"]), eps=cfg.eps, max_len=max_len)
    torch.cuda.synchronize()
    for k, v in (("y", y), ("residual", h["residual"]), ("q", h["q"]), ("out", out),
                 ("k_cache", kc), ("v_cache", vc)):
        same(v, r[k], k)

    big = CONFIGS["serving_small"]
    inp = W.make_inputs(big)
    B, Hq, D = inp["q"].shape
    max_len = int(inp["lens"].max())
    assert dsa.decode_step_path(B, Hq, big.Hkv, D, max_len) == dsa.STEP_STREAM
    d = {k: on_dev(inp[k]) for k in ("x", "residual", "norm_w", "k_new", "v_new", "pos", "lens",
                                     "k_cache", "v_cache", "q_norm_w", "k_norm_w")}
    ws = dsa.alloc_workspace(B, Hq, big.Hkv, D, max_len)
    with pytest.raises(dsa.DecAttnError, match="q must be device memory"):
        dsa.decode_step(d["x"], d["residual"], d["norm_w"], torch.empty_like(d["x"]),
                        pinned(inp["q"]), d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                        d["pos"], d["lens"], torch.empty(B, Hq, D, dtype=torch.bfloat16,
                                                         device=DEV),
                        ws, theta=big.theta, layout=big.layout, q_norm_w=d["q_norm_w"],
                        k_norm_w=d["k_norm_w"], eps=big.eps, max_len=max_len)


def test_sublayer_with_host_arguments():
    """The attention sublayer with x, the residual, pos, lens and out in pinned host
    memory: the same kernels, so the same bits as the device-resident call."""
    cfg = W.small_variant(W.SERVING_MIX, B=12, max_len=300)
    inp = W.make_inputs(cfg)
    wts = W.make_projection_weights(cfg)
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    T_cap = inp["t_cap"]
    max_len = int(inp["lens"].max())
    common = dict(norm_w=inp["norm_w"].to(DEV), w_qkv=wts["w_qkv"].to(DEV),
                  w_o=wts["w_o"].to(DEV), theta=cfg.theta, layout=cfg.layout,
                  q_norm_w=on_dev(inp["q_norm_w"]), k_norm_w=on_dev(inp["k_norm_w"]),
                  eps=cfg.eps, max_len=max_len)
    nbytes = dsa.sublayer_workspace_bytes(B, H, Hq, Hkv, D, max_len)
    runs = []
    for host in (False, True):
        put = pinned if host else on_dev
        r = put(inp["residual"])
        out = (torch.empty(B, H, dtype=torch.bfloat16, pin_memory=True) if host
               else torch.empty(B, H, dtype=torch.bfloat16, device=DEV))
        kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
        dsa.attn_sublayer(put(inp["x"]), r, k_cache=kc, v_cache=vc, pos=put(inp["pos"]),
                          lens=put(inp["lens"]), out=out, workspace=ws, **common)
        torch.cuda.synchronize()
        assert dsa.device_errors(ws) == 0
        runs.append((out, r, kc, vc))
    for k, a, b in zip(("out", "residual", "k_cache", "v_cache"), runs[0], runs[1]):
        same(b, a, k)
    assert T_cap >= max_len


def test_graph_branch_with_copies():
    """A StepGraph branch with copies of its own: the RMSNorm half of the step runs on a
    second stream from device buffers filled by the branch's copy in, and its results
    go back by the branch's copy out, while the attention half runs zero-copy."""
    cfg = CONFIGS["serving_small"]
    inp = W.make_inputs(cfg)
    r = device_step(cfg, inp)
    hs = HostStep(cfg, inp)
    x_d = torch.empty(tuple(inp["x"].shape), dtype=torch.bfloat16, device=DEV)
    res_d = torch.empty_like(x_d)
    y_d = torch.empty_like(x_d)

    def k1_dev():
        dsa.rmsnorm_residual(x_d, hs.d["norm_w"], residual=res_d, eps=cfg.eps, out=y_d)

    br = dsa.GraphBranch(k1_dev, copies_in=[(hs.h["x"], x_d), (hs.h["residual"], res_d)],
                         copies_out=[(y_d, hs.h["y"]), (res_d, hs.h["residual"])])
    g = dsa.StepGraph(prologue=hs.k2, step=hs.attn, branches=[br])
    hs.h["residual"].copy_(inp["residual"])  # the constructor's eager run updated it
    hs.h["y"].zero_()
    hs.h["out"].zero_()
    g.replay()
    torch.cuda.synchronize()
    check_against(r, hs, inp)
