"""Randomised shapes through the whole step and the attention call (GPU only).

Each case draws a batch, head counts, head_dim, RoPE layout, QK-norm, lengths
(including 0 for the attention call, 1, tile edges and T_cap) and a forced number of
split-pass CTAs, runs the CUDA path and checks every stage against the oracle on
that stage's own inputs.
"""
import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W
from oracle import decode_ref as O
from tol import check_float, check_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f64(t):
    return t.double().cpu().numpy()


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    D = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 24))
    T = int(rng.choice([1, 7, 64, 127, 128, 129, 300, 1500, 5000]))
    lens = rng.integers(1, T + 1, size=B)
    lens[rng.random(B) < 0.2] = T
    lens[rng.random(B) < 0.1] = 1
    cfg = W.BlockConfig(f"fuzz{seed}", B=B, hidden=int(rng.choice([64, 256, 1024])), Hq=G * Hkv,
                        Hkv=Hkv, D=D, theta=float(rng.choice([1e4, 5e5, 1e6])),
                        layout=str(rng.choice(["neox", "interleaved"])), qk_norm=bool(rng.random() < 0.5),
                        lens_kind="list", lens_args=tuple(int(x) for x in lens), t_cap=T, seed=seed)
    parts = int(rng.choice([0, 0, 1, 2, 5, 37, 152, 400]))
    if rng.random() < 0.4:  # blocks of >= 4096 rows: large pieces plus claimed small ones
        rows = Hkv * int(lens.sum())
        parts = max(1, rows // int(rng.integers(4096, 20000)))
    return cfg, parts


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_step(seed):
    cfg, parts = _case(seed)
    inp = W.make_inputs(cfg)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    max_len = int(inp["lens"].max())
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len, parts)
    y, out, resid, q = torch.empty_like(d["x"]), torch.empty_like(d["q"]), d["residual"].clone(), d["q"].clone()
    dsa.decode_step(d["x"], resid, d["norm_w"], y, q, d["k_new"], d["v_new"], d["k_cache"],
                    d["v_cache"], d["pos"], d["lens"], out, ws, theta=cfg.theta, layout=cfg.layout,
                    q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len,
                    num_parts=parts)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]), cfg.eps)
    check_float(f64(y), y_ref, "y")
    check_ulp(f64(resid), s_ref, "residual")
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    check_float(f64(q), O.qknorm_rope(f64(inp["q"]), qn, inp["pos"].numpy(), cfg.theta, cfg.layout,
                                      cfg.eps), "q")
    ref = O.gqa_decode_attention(f64(q), f64(d["k_cache"]), f64(d["v_cache"]), inp["lens"].numpy())
    check_float(f64(out), ref, f"out (parts={parts})")


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_attention_with_empty_sequences(seed):
    cfg, parts = _case(100 + seed)
    inp = W.make_inputs(cfg)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    lens = inp["lens"].numpy().copy()
    for b in range(cfg.B):
        p = int(inp["pos"][b])
        kc[b, :, p] = inp["k_new"][b]
        vc[b, :, p] = inp["v_new"][b]
    zero = np.random.default_rng(seed).random(cfg.B) < 0.3
    lens[zero] = 0
    lens_t = torch.from_numpy(lens.astype(np.int32)).to(DEV)
    max_len = int(max(lens.max(), 0))
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len, parts)
    out = dsa.gqa_decode_attn(inp["q"].to(DEV), kc.to(DEV), vc.to(DEV), lens_t, max_len=max_len,
                              workspace=ws, num_parts=parts)
    torch.cuda.synchronize()
    ref = O.gqa_decode_attention(f64(inp["q"]), f64(kc), f64(vc), lens)
    check_float(f64(out), ref, f"attention (parts={parts})")
    assert dsa.device_errors(ws) == 0


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_attention_one_launch(seed):
    """Short contexts with the split left to the library: the attention call's one-launch
    path, with and without a window, empty sequences included."""
    rng = np.random.default_rng(5000 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 8]))
    D = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 64 // Hkv + 1))
    T = int(rng.choice([1, 2, 15, 16, 17, 100, 513, 1024]))
    lens = rng.integers(0, T + 1, size=B)
    lens[rng.random(B) < 0.3] = T
    window = int(rng.choice([0, 0, 1, 5, 64, 2000]))
    cfg = W.BlockConfig(f"fuzz_small{seed}", B=B, hidden=64, Hq=G * Hkv, Hkv=Hkv, D=D, theta=1e4,
                        layout="neox", qk_norm=False, lens_kind="list",
                        lens_args=tuple(max(1, int(x)) for x in lens), t_cap=T, seed=seed)
    inp = W.make_inputs(cfg)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    for b in range(B):  # the new token's slot, as the append leaves it
        p = int(inp["pos"][b])
        kc[b, :, p] = inp["k_new"][b]
        vc[b, :, p] = inp["v_new"][b]
    max_len = int(lens.max()) if lens.max() > 0 else 0
    assert dsa.decode_step_launches(B, G * Hkv, Hkv, D, max_len, window) == 1
    lens_t = torch.from_numpy(lens.astype(np.int32)).to(DEV)
    ws = dsa.alloc_workspace(B, G * Hkv, Hkv, D, max_len)
    out = dsa.gqa_decode_attn(inp["q"].to(DEV), kc.to(DEV), vc.to(DEV), lens_t, max_len=max_len,
                              workspace=ws, window=window)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    ref = O.gqa_decode_attention(f64(inp["q"]), f64(kc), f64(vc), lens, window=window or None)
    check_float(f64(out), ref, f"one-launch attention (window {window})")
