"""dec_gqa_decode_attn_noalloc: attention with the library's static scratch (GPU only).

The allocation-free call serves callers that cannot allocate device memory when
they run attention (inside an allocator hook or host callback, or in a runtime that
owns every allocation). It runs the same kernels as the regular call with a
caller-provided workspace, so on the same inputs and the same split it must give
the same bits, call after call, even though every call reuses one static buffer
that keeps the previous call's contents; and both must match the fp64 oracle. It
must not allocate: once the library's module is loaded on the device, neither
torch's allocator nor the driver's free-memory count moves across a call. This
file runs last so a failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W
from oracle import decode_ref as O
from tol import check_float

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20
LEN_CLAMPED = 0x1


def _inputs(cfg):
    inp = W.make_inputs(cfg)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    for b in range(cfg.B):
        p = int(inp["pos"][b])
        kc[b, :, p] = inp["k_new"][b]
        vc[b, :, p] = inp["v_new"][b]
    return {"q": inp["q"].cuda(), "k": kc.cuda(), "v": vc.cuda(), "lens": inp["lens"].cuda(),
            "max_len": int(inp["lens"].max()), "t_cap": inp["t_cap"],
            "ref": O.gqa_decode_attention(inp["q"].double().numpy(), kc.double().numpy(),
                                          vc.double().numpy(), inp["lens"].numpy())}


def _noalloc(L, t, out, Hkv, num_parts=0, err=None):
    B, Hq, D = t["q"].shape
    return L.dec_gqa_decode_attn_noalloc(
        ctypes.c_void_p(t["q"].data_ptr()), ctypes.c_void_p(t["k"].data_ptr()),
        ctypes.c_void_p(t["v"].data_ptr()), ctypes.c_void_p(t["lens"].data_ptr()),
        ctypes.c_void_p(out.data_ptr()), B, Hq, Hkv, D, t["t_cap"], t["max_len"], 0.0, num_parts,
        ctypes.c_void_p(0 if err is None else err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = {
    # the split pass and its merge (more than 1024 attended rows)
    "serving_split": (W.small_variant(W.SERVING_MIX, B=24, max_len=1500, seed=1), 0),
    "llama_split": (W.small_variant(W.LLAMA3_BATCHED, B=5, max_len=2000, seed=2), 0),
    # a split count given by the caller
    "llama_forced_parts": (W.small_variant(W.LLAMA3_BATCHED, B=5, max_len=2000, seed=3), 37),
    # a short context: the one-launch attention kernel (split and merge in one cluster)
    "qwen_one_launch": (W.QWEN3_512, 0),
    "serving_one_launch": (W.small_variant(W.SERVING_MIX, B=12, max_len=700, seed=4), 0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_call_twice_in_a_row(name):
    cfg, parts = CASES[name]
    L = dsa.lib()
    t = _inputs(cfg)
    path = dsa.decode_step_path(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, t["max_len"])
    assert path == (dsa.STEP_SHORT if name.endswith("one_launch") else dsa.STEP_STREAM)
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, t["max_len"], parts)
    ref = dsa.gqa_decode_attn(t["q"], t["k"], t["v"], t["lens"], max_len=t["max_len"],
                              workspace=ws, num_parts=parts)
    outs = [torch.full_like(t["q"], float("nan")) for _ in range(3)]
    err = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    # first call: may load the library's module (and with it the static scratch)
    assert _noalloc(L, t, outs[0], cfg.Hkv, parts, err) == 0, L.dec_last_error().decode()
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for out in outs[1:]:  # each call reuses the scratch the previous one left behind
        assert _noalloc(L, t, out, cfg.Hkv, parts, err) == 0, L.dec_last_error().decode()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    ref_bits = ref.view(torch.int16).cpu()
    for out in outs:
        assert torch.equal(out.view(torch.int16).cpu(), ref_bits), f"{name}: not bit-identical"
        check_float(out.double().cpu().numpy(), t["ref"], f"{name} against the oracle")


def test_noalloc_reports_its_own_device_errors():
    """A length past the cache is clamped and flagged; the next clean call reports 0."""
    L = dsa.lib()
    cfg = W.small_variant(W.SERVING_MIX, B=8, max_len=1500, seed=5)
    t = _inputs(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = dict(t, lens=t["lens"].clone())
    bad["lens"][3] = t["t_cap"] + 9  # clamped to T_cap on the device (documented)
    out = torch.empty_like(t["q"])
    assert _noalloc(L, bad, out, cfg.Hkv, 0, err) == 0, L.dec_last_error().decode()
    torch.cuda.synchronize()
    assert int(err.item()) & LEN_CLAMPED
    assert _noalloc(L, t, out, cfg.Hkv, 0, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_float(out.double().cpu().numpy(), t["ref"], "after a clamped call")


def _exactly_at_the_limit(L, Hq, Hkv, D, T):
    """(num_parts, B) whose workspace is exactly the 4 MiB of the static scratch."""
    for parts in range(152, 0, -1):
        lo, hi = 1, 1 << 14
        while lo < hi:  # the largest B that fits; the workspace grows with B
            mid = (lo + hi + 1) // 2
            if L.dec_attn_workspace_bytes(mid, Hq, Hkv, D, T, parts) <= SCRATCH_BYTES:
                lo = mid
            else:
                hi = mid - 1
        if L.dec_attn_workspace_bytes(lo, Hq, Hkv, D, T, parts) == SCRATCH_BYTES:
            return parts, lo
    raise AssertionError("no split count puts this shape exactly at the limit")


def test_noalloc_at_the_scratch_limit():
    """A shape whose workspace is exactly the 4 MiB buffer runs and matches the
    workspace call bit for bit; one more sequence is refused before anything is
    enqueued."""
    L = dsa.lib()
    Hq, Hkv, D, T = 16, 4, 128, 40
    parts, B = _exactly_at_the_limit(L, Hq, Hkv, D, T)
    assert L.dec_attn_workspace_bytes(B + 1, Hq, Hkv, D, T, parts) > SCRATCH_BYTES
    rng = np.random.default_rng(11)
    lens_list = tuple(int(x) for x in rng.integers(1, T + 1, size=B))
    cfg = W.BlockConfig("at_limit", B=B, hidden=256, Hq=Hq, Hkv=Hkv, D=D, theta=1e4,
                        layout="neox", qk_norm=False, lens_kind="list", lens_args=lens_list,
                        t_cap=T, seed=12)
    t = _inputs(cfg)
    t["max_len"] = T
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, T, parts)
    ref = dsa.gqa_decode_attn(t["q"], t["k"], t["v"], t["lens"], max_len=T, workspace=ws,
                              num_parts=parts)
    out = torch.full_like(t["q"], float("nan"))
    assert _noalloc(L, t, out, Hkv, parts) == 0, L.dec_last_error().decode()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    check_float(out.double().cpu().numpy(), t["ref"], "at the scratch limit")
    # one more sequence: refused, nothing launched
    q1 = torch.zeros(B + 1, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(B + 1, Hkv, T, D, dtype=torch.bfloat16, device="cuda")
    big = {"q": q1, "k": kc, "v": kc.clone(), "lens": torch.ones(B + 1, dtype=torch.int32,
                                                                   device="cuda"),
           "t_cap": T, "max_len": T}
    out1 = torch.zeros_like(q1)
    st = _noalloc(L, big, out1, Hkv, parts)
    assert st == 3 and "4 MiB" in L.dec_last_error().decode()
    torch.cuda.synchronize()
    assert torch.all(out1 == 0)


def test_noalloc_rejects_bad_arguments_without_launching():
    """A refused call (a non-finite scale, a misaligned output, a bad head count)
    returns its status and launches nothing: the output keeps its contents."""
    L = dsa.lib()
    cfg = W.small_variant(W.SERVING_MIX, B=8, max_len=1500, seed=6)
    t = _inputs(cfg)
    out = torch.full_like(t["q"], 3.0)
    B, Hq, D = t["q"].shape
    args = [ctypes.c_void_p(t["q"].data_ptr()), ctypes.c_void_p(t["k"].data_ptr()),
            ctypes.c_void_p(t["v"].data_ptr()), ctypes.c_void_p(t["lens"].data_ptr()),
            ctypes.c_void_p(out.data_ptr()), B, Hq, cfg.Hkv, D, t["t_cap"], t["max_len"], 0.0, 0,
            ctypes.c_void_p(0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)]
    bad_scale = list(args)
    bad_scale[11] = float("inf")
    assert L.dec_gqa_decode_attn_noalloc(*bad_scale) == 1
    bad_heads = list(args)
    bad_heads[7] = 3  # Hq = 16 is not a multiple of 3
    assert L.dec_gqa_decode_attn_noalloc(*bad_heads) == 1
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    bad_err = list(args)
    bad_err[13] = ctypes.c_void_p(err.data_ptr() + 2)  # a misaligned error word
    assert L.dec_gqa_decode_attn_noalloc(*bad_err) == 1
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    # B = 0 enqueues nothing either (the error word is left as it was)
    err7 = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    empty = dict(t, q=t["q"][:0])
    assert _noalloc(L, empty, out, cfg.Hkv, 0, err7) == 0
    torch.cuda.synchronize()
    assert int(err7.item()) == 7
