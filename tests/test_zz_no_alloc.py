"""dec_gqa_decode_attn_noalloc: attention with the library's static scratch (GPU only).

The allocation-free call serves callers that cannot allocate device memory when
they run attention (inside an allocator hook or host callback, or in a runtime that
owns every allocation). It must give the same result as the regular call with a
caller-provided workspace, call after call, even though every call reuses one
static buffer that keeps the previous call's contents. This file runs last so a
failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W
from tol import check_float

pytestmark = pytest.mark.gpu


def _inputs(cfg):
    inp = W.make_inputs(cfg)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    for b in range(cfg.B):
        p = int(inp["pos"][b])
        kc[b, :, p] = inp["k_new"][b]
        vc[b, :, p] = inp["v_new"][b]
    return {"q": inp["q"].cuda(), "k": kc.cuda(), "v": vc.cuda(), "lens": inp["lens"].cuda(),
            "max_len": int(inp["lens"].max()), "t_cap": inp["t_cap"]}


def _noalloc(L, t, out, Hkv):
    B, Hq, D = t["q"].shape
    st = L.dec_gqa_decode_attn_noalloc(
        ctypes.c_void_p(t["q"].data_ptr()), ctypes.c_void_p(t["k"].data_ptr()),
        ctypes.c_void_p(t["v"].data_ptr()), ctypes.c_void_p(t["lens"].data_ptr()),
        ctypes.c_void_p(out.data_ptr()), B, Hq, Hkv, D, t["t_cap"], t["max_len"], 0.0, 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_workspace_call_twice_in_a_row():
    L = dsa.lib()
    cfgs = [W.small_variant(W.SERVING_MIX, B=24, max_len=1500, seed=1),
            W.small_variant(W.LLAMA3_BATCHED, B=5, max_len=2000, seed=2)]
    for cfg in cfgs:
        t = _inputs(cfg)
        ref = dsa.gqa_decode_attn(t["q"], t["k"], t["v"], t["lens"], max_len=t["max_len"])
        for _ in range(2):  # the second call reuses the scratch the first one left behind
            out = torch.full_like(t["q"], float("nan"))
            st = _noalloc(L, t, out, cfg.Hkv)
            assert st == 0, L.dec_last_error().decode()
            torch.cuda.synchronize()
            check_float(out.double().cpu().numpy(), ref.double().cpu().numpy(), cfg.name)


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    L = dsa.lib()
    B, Hq, Hkv, D, T = 2048, 64, 8, 128, 16
    need = L.dec_attn_workspace_bytes(B, Hq, Hkv, D, T, 0)
    assert need > (4 << 20)
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(B, Hkv, T, D, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    t = {"q": q, "k": kc, "v": kc, "lens": lens, "t_cap": T, "max_len": T}
    st = _noalloc(L, t, out, Hkv)
    assert st == 3 and "4 MiB" in L.dec_last_error().decode()
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched
