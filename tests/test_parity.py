"""CUDA path against the CPU oracle on identical seeded bf16 inputs (GPU only).

Each kernel is compared on its own inputs (stage by stage), element by element at
sizes the oracle finishes in seconds and on sampled outputs at the full workload
sizes, with the tolerances of tests/tol.py.
"""
import math

import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W
from oracle import decode_ref as O
from tol import check_float, check_ulp

pytestmark = pytest.mark.gpu

DEV = "cuda"
LN2 = math.log(2.0)

SMALL = {
    "tiny": W.TINY,
    "qwen3_ctx128": W.QWEN3_128,
    "qwen3_ctx512": W.QWEN3_512,
    "llama3_small": W.small_variant(W.LLAMA3_BATCHED, B=6, max_len=900),
    "long_small": W.small_variant(W.LONG_CONTEXT, max_len=3000),
    "serving_small": W.small_variant(W.SERVING_MIX, B=40, max_len=700),
}


def f64(t):
    return t.double().cpu().numpy()


def dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def bits(t):
    return t.view(torch.int16).cpu().numpy()


def with_new_token(inp):
    """Caches with the new token's raw K/V in slot pos_b (the attention stage's input)."""
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    for b in range(kc.shape[0]):
        p = int(inp["pos"][b])
        kc[b, :, p] = inp["k_new"][b]
        vc[b, :, p] = inp["v_new"][b]
    return kc, vc


# ---------------------------------------------------------------- K1 ---
@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("with_residual", [True, False])
def test_rmsnorm_residual(name, with_residual):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, with_cache=False)
    d = dev(inp)
    res = d["residual"].clone() if with_residual else None
    y = dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=res, eps=cfg.eps)
    torch.cuda.synchronize()
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]) if with_residual else None,
                                      f64(inp["norm_w"]), cfg.eps)
    check_float(f64(y), y_ref, f"{name} y")
    if with_residual:
        check_ulp(f64(res), s_ref, f"{name} residual", ulps=1.0)


def test_rmsnorm_wide_rows():
    cfg = W.LLAMA3_BATCHED.replace(B=3, hidden=16384, seed=5)
    inp = W.make_inputs(cfg, with_cache=False)
    d = dev(inp)
    res = d["residual"].clone()
    y = dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=res, eps=cfg.eps)
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]), cfg.eps)
    check_float(f64(y), y_ref, "hidden 16384")
    check_ulp(f64(res), s_ref, "hidden 16384 residual")


# ---------------------------------------------------------------- K2 ---
def _append_check(cfg, inp, label, freq=(None, None)):
    """K2 against the oracle; ``freq`` = (the GPU's RoPE table, the oracle's), or none."""
    d = dev(inp)
    q = d["q"].clone()
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.qknorm_rope_kv_append(q, d["k_new"], d["v_new"], kc, vc, d["pos"], cfg.theta, cfg.layout,
                              d["q_norm_w"], d["k_norm_w"], cfg.eps, error_word=err,
                              inv_freq=freq[0])
    torch.cuda.synchronize()
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    kn = None if inp["k_norm_w"] is None else f64(inp["k_norm_w"])
    pos = inp["pos"].numpy()
    q_rot = O.qknorm_rope(f64(inp["q"]), qn, pos, cfg.theta, cfg.layout, cfg.eps, freq[1])
    k_rot = O.qknorm_rope(f64(inp["k_new"]), kn, pos, cfg.theta, cfg.layout, cfg.eps, freq[1])
    check_float(f64(q), q_rot, f"{label} q")
    kb, vb = bits(kc), bits(vc)
    kb0, vb0 = bits(inp["k_cache"]), bits(inp["v_cache"])
    new_k = np.stack([f64(kc[b, :, int(pos[b])]) for b in range(cfg.B)])
    check_ulp(new_k, k_rot, f"{label} appended k", ulps=1.0)
    for b in range(cfg.B):
        p = int(pos[b])
        assert np.array_equal(vb[b, :, p], bits(inp["v_new"])[b]), "v slot is not a bit copy"
        mask = np.ones(kb.shape[2], bool)
        mask[p] = False
        assert np.array_equal(kb[b][:, mask], kb0[b][:, mask]), "other K slots changed"
        assert np.array_equal(vb[b][:, mask], vb0[b][:, mask]), "other V slots changed"
    assert int(err.item()) == 0


@pytest.mark.parametrize("name", list(SMALL))
def test_qknorm_rope_append(name):
    cfg = SMALL[name]
    _append_check(cfg, W.make_inputs(cfg), name)


@pytest.mark.parametrize("layout", ["neox", "interleaved"])
@pytest.mark.parametrize("qk_norm", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_append_layouts(layout, qk_norm, D):
    cfg = W.BlockConfig("append_mix", B=5, hidden=256, Hq=8, Hkv=2, D=D, theta=5e5, layout=layout,
                        qk_norm=qk_norm, lens_kind="list", lens_args=(1, 2, 900, 131072, 77777),
                        t_cap=131072, seed=3)
    inp = W.make_inputs(cfg, with_cache=False)
    T = 131072
    inp["k_cache"] = W.nan_bf16((cfg.B, cfg.Hkv, T, D))
    inp["v_cache"] = W.nan_bf16((cfg.B, cfg.Hkv, T, D))
    _append_check(cfg, inp, f"{layout}/{qk_norm}/{D}")


@pytest.mark.parametrize("B,Hq,Hkv,layout", [(200, 12, 4, "interleaved"),  # 2 heads a warp
                                              (160, 16, 4, "neox"),          # 3 heads a warp
                                              (400, 32, 8, "neox")])         # 4, a ragged last CTA
def test_append_several_heads_per_warp(B, Hq, Hkv, layout):
    """Batches large enough that each warp of the rotation kernel takes several heads
    (K2 alone, and K2 inside the decode step with its RMSNorm rows), against the oracle."""
    cfg = W.BlockConfig("append_wide", B=B, hidden=256, Hq=Hq, Hkv=Hkv, D=128, theta=1e4,
                        layout=layout, qk_norm=True, lens_kind="uniform", lens_args=(1, 96),
                        t_cap=96, seed=7)
    inp = W.make_inputs(cfg)
    _append_check(cfg, inp, f"B={B} Hq={Hq} Hkv={Hkv}")
    st = _step(cfg, inp)
    pos = inp["pos"].numpy()
    q_rot = O.qknorm_rope(f64(inp["q"]), f64(inp["q_norm_w"]), pos, cfg.theta, cfg.layout, cfg.eps)
    k_rot = O.qknorm_rope(f64(inp["k_new"]), f64(inp["k_norm_w"]), pos, cfg.theta, cfg.layout,
                          cfg.eps)
    check_float(f64(st["q"]), q_rot, "step q")
    new_k = np.stack([f64(st["k_cache"][b, :, int(pos[b])]) for b in range(cfg.B)])
    check_ulp(new_k, k_rot, "step appended k", ulps=1.0)
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]),
                                      cfg.eps)
    check_float(f64(st["y"]), y_ref, "step y")


def test_append_skips_bad_positions():
    cfg = W.small_variant(W.QWEN3_128, B=3, max_len=16)
    inp = W.make_inputs(cfg)
    d = dev(inp)
    pos = torch.tensor([0, 16, -1], dtype=torch.int32, device=DEV)  # T_cap = 16
    q = d["q"].clone()
    kc = d["k_cache"].clone()
    vc = d["v_cache"].clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.qknorm_rope_kv_append(q, d["k_new"], d["v_new"], kc, vc, pos, cfg.theta, cfg.layout,
                              d["q_norm_w"], d["k_norm_w"], cfg.eps, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dsa.DEVERR_POS_SKIPPED
    assert torch.equal(q[1:].view(torch.int16), d["q"][1:].view(torch.int16))
    assert torch.equal(kc[1:].view(torch.int16), d["k_cache"][1:].view(torch.int16))


# ---------------------------------------------------------- K3 + K4 ---
def _attn_ref(inp, kc, vc, lens, scale=None):
    return O.gqa_decode_attention(f64(inp["q"]), f64(kc), f64(vc), lens, scale)


def _run_attn(d, kc, vc, lens_t, max_len, num_parts=0, scale=0.0):
    B, Hq, D = d["q"].shape
    Hkv = kc.shape[1]
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, max_len, num_parts)
    out = dsa.gqa_decode_attn(d["q"], kc, vc, lens_t, max_len=max_len, workspace=ws,
                              num_parts=num_parts, scale=scale)
    torch.cuda.synchronize()
    return out, ws


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("num_parts", [0, 1, 3, 1000])
def test_gqa_decode_attn(name, num_parts):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    d = dev(inp)
    lens = inp["lens"].numpy()
    out, ws = _run_attn(d, kc.to(DEV), vc.to(DEV), d["lens"], int(lens.max()), num_parts)
    check_float(f64(out), _attn_ref(inp, kc, vc, lens), f"{name} parts={num_parts}")
    assert dsa.device_errors(ws) == 0


def _sched(total, parts):
    """The split pass's piece boundaries (see PieceSched in the CUDA sources)."""
    blk = max(64, -(-total // parts))
    if blk >= 4096:
        big = blk * 800 // 1000
        cs = -(-(blk - big) // 4)
    else:
        big, cs = blk, 1

    def start(i):
        c, j = divmod(i, 5)
        r = c * blk if j == 0 else c * blk + big + (j - 1) * cs
        return min(r, (c + 1) * blk, total)

    def piece_of(row):
        c, off = divmod(row, blk)
        return 5 * c if off < big else 5 * c + 1 + (off - big) // cs
    return start, piece_of


def _slots(B, Hkv, parts):
    return 5 * parts + B * Hkv


def _partition(lens, Hkv, parts):
    """The split pass's cut of the (b, g, t) row stream: {(b, g): [(piece, t0, t1), ...]}."""
    lens = [int(x) for x in lens]
    total = Hkv * sum(lens)
    start, piece_of = _sched(total, parts)
    out = {}
    s = 0
    for b, L in enumerate(lens):
        for g in range(Hkv):
            e = s + L
            lst = []
            if L > 0:
                for c in range(piece_of(s), piece_of(e - 1) + 1):
                    lo, hi = max(s, start(c)), min(e, start(c + 1))
                    if lo < hi:  # empty pieces (small pieces of unsplit blocks) hold nothing
                        lst.append((c, lo - s, hi - s))
            out[(b, g)] = lst
            s = e
    return out


@pytest.mark.parametrize("name", ["llama3_small", "serving_small", "long_small"])
@pytest.mark.parametrize("num_parts", [5, 64])
def test_split_partials(name, num_parts):
    """The split pass's partials against oracle partials on the same token ranges."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    d = dev(inp)
    lens = inp["lens"].numpy()
    B, Hq, Hkv, D, G = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.G
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, int(lens.max()), num_parts)
    dsa.gqa_decode_split(d["q"], kc.to(DEV), vc.to(DEV), d["lens"], ws, max_len=int(lens.max()),
                         num_parts=num_parts)
    torch.cuda.synchronize()
    slots = _slots(B, Hkv, num_parts)
    body = ws[dsa.WORKSPACE_HEADER_BYTES:].view(torch.float32).cpu().numpy()
    o_ws = body[:slots * G * D].reshape(slots, G, D)
    lse_ws = body[slots * G * D: slots * G * D + slots * G].reshape(slots, G)
    qf, kf, vf = f64(inp["q"]), f64(kc), f64(vc)
    scale = 1.0 / math.sqrt(D)
    n = 0
    for (b, g), lst in _partition(lens, Hkv, num_parts).items():
        for (c, t0, t1) in lst:
            slot = c + b * Hkv + g
            for hh in range(G):
                o_ref, lse_ref = O.attention_partial(qf[b, g * G + hh], kf[b, g, t0:t1], vf[b, g, t0:t1], scale)
                check_float(o_ws[slot, hh], o_ref, f"partial o {(b, g, c, hh)}", abs_tol=1e-3, rel_rms=1e-4)
                assert abs(lse_ws[slot, hh] * LN2 - lse_ref) <= 1e-4 * max(1.0, abs(lse_ref)), (b, g, c, hh)
                n += 1
    assert n > 0


@pytest.mark.parametrize("num_parts", [1, 7, 40])
def test_merge_alone(num_parts):
    """The merge pass fed with oracle partials written into the workspace layout."""
    cfg = SMALL["serving_small"]
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    lens = inp["lens"].numpy()
    B, Hq, Hkv, D, G = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.G
    slots = _slots(B, Hkv, num_parts)
    o_ws = np.zeros((slots, G, D), np.float32)
    lse_ws = np.full((slots, G), np.nan, np.float32)
    qf, kf, vf = f64(inp["q"]), f64(kc), f64(vc)
    scale = 1.0 / math.sqrt(D)
    for (b, g), lst in _partition(lens, Hkv, num_parts).items():
        for (c, t0, t1) in lst:
            for hh in range(G):
                o, lse = O.attention_partial(qf[b, g * G + hh], kf[b, g, t0:t1], vf[b, g, t0:t1], scale)
                o_ws[c + b * Hkv + g, hh] = o
                lse_ws[c + b * Hkv + g, hh] = lse / LN2
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, int(lens.max()), num_parts)
    body = torch.from_numpy(np.concatenate([o_ws.ravel(), lse_ws.ravel()]).view(np.uint8))
    ws[dsa.WORKSPACE_HEADER_BYTES:dsa.WORKSPACE_HEADER_BYTES + body.numel()] = body.to(DEV)
    # the sequence offsets the split pass would have left behind
    off = (dsa.WORKSPACE_HEADER_BYTES + body.numel() + 15) // 16 * 16
    prefix = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ws[off:off + 4 * (B + 1)] = torch.from_numpy(prefix.view(np.uint8)).to(DEV)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=DEV)
    dsa.split_merge(ws, inp["lens"].to(DEV), out, Hkv, inp["t_cap"], max_len=int(lens.max()),
                    num_parts=num_parts)
    torch.cuda.synchronize()
    check_float(f64(out), _attn_ref(inp, kc, vc, lens), f"merge parts={num_parts}")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_group_sizes_and_edges(G, D):
    lens_list = (1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 200, 0, 333)
    Hkv = 2
    cfg = W.BlockConfig("edges", B=len(lens_list), hidden=256, Hq=G * Hkv, Hkv=Hkv, D=D, theta=1e4,
                        layout="neox", qk_norm=False, lens_kind="list", lens_args=lens_list,
                        t_cap=333, seed=G * 10 + D)
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    for b, L in enumerate(lens_list):  # a zero-length sequence has no new token either
        if L == 0:
            kc[b].fill_(float("nan"))
            vc[b].fill_(float("nan"))
    lens = inp["lens"].numpy()
    d = dev(inp)
    for parts in (0, 2, 9):
        out, ws = _run_attn(d, kc.to(DEV), vc.to(DEV), d["lens"], 333, parts)
        ref = _attn_ref(inp, kc, vc, lens)
        check_float(f64(out), ref, f"G={G} D={D} parts={parts}")
        assert torch.all(out[lens_list.index(0)] == 0)


def test_large_batch_prefix_scan():
    """More sequences than threads in a CTA, many of them empty or one token long."""
    rng = np.random.default_rng(7)
    lens_list = tuple(int(x) for x in rng.choice([0, 1, 2, 5, 70, 300], size=700))
    cfg = W.BlockConfig("many", B=700, hidden=256, Hq=8, Hkv=2, D=128, theta=1e4, layout="neox",
                        qk_norm=False, lens_kind="list", lens_args=lens_list, t_cap=300, seed=11)
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    lens = inp["lens"].numpy()
    for b in np.nonzero(lens == 0)[0]:
        kc[b].fill_(float("nan"))
        vc[b].fill_(float("nan"))
    d = dev(inp)
    out, ws = _run_attn(d, kc.to(DEV), vc.to(DEV), d["lens"], 300, 0)
    check_float(f64(out), _attn_ref(inp, kc, vc, lens), "B=700")


def test_peaked_softmax_and_scale():
    cfg = W.small_variant(W.LONG_CONTEXT, max_len=2500)
    inp = W.make_inputs(cfg)
    inp["q"] = (inp["q"].float() * 6.0).to(torch.bfloat16)  # logits up to ~+-60
    kc, vc = with_new_token(inp)
    d = dev(inp)
    lens = inp["lens"].numpy()
    out, _ = _run_attn(d, kc.to(DEV), vc.to(DEV), d["lens"], 2500, 0)
    check_float(f64(out), _attn_ref(inp, kc, vc, lens), "peaked")
    out, _ = _run_attn(d, kc.to(DEV), vc.to(DEV), d["lens"], 2500, 0, scale=0.01)
    check_float(f64(out), _attn_ref(inp, kc, vc, lens, scale=0.01), "scale 0.01")


def test_lengths_clamped_and_flagged():
    cfg = W.small_variant(W.QWEN3_128, B=2, max_len=64)
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    d = dev(inp)
    lens_t = torch.tensor([64, 500], dtype=torch.int32, device=DEV)  # 500 > T_cap = 64
    kc[1] = torch.randn(kc[1].shape).to(torch.bfloat16)
    vc[1] = torch.randn(vc[1].shape).to(torch.bfloat16)
    out, ws = _run_attn(d, kc.to(DEV), vc.to(DEV), lens_t, 64, 0)
    assert dsa.device_errors(ws) & dsa.DEVERR_LEN_CLAMPED
    check_float(f64(out), _attn_ref(inp, kc, vc, np.array([64, 64])), "clamped")


def test_bounded_wait_reports_instead_of_hanging():
    """A pipeline wait that never completes gives up, sets the error bit, and the
    context keeps working afterwards."""
    import time
    L = dsa.lib()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert L.dec_diag_wait_timeout(ctypes_ptr(err), dsa._stream()) == 0
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert int(err.item()) & dsa.DEVERR_WAIT_TIMEOUT
    assert 0.9 < took < 10.0, took
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum()) == 8.0  # still usable
    print(f"bounded wait gave up after {took:.3f} s")


def ctypes_ptr(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


def test_empty_batch_and_all_empty():
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=DEV)
    kc = torch.empty(0, 2, 16, 128, dtype=torch.bfloat16, device=DEV)
    lens = torch.empty(0, dtype=torch.int32, device=DEV)
    ws = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    out = dsa.gqa_decode_attn(q, kc, kc.clone(), lens, max_len=0, workspace=ws)
    assert out.shape == (0, 8, 128)
    q = torch.randn(3, 8, 128, device=DEV).to(torch.bfloat16)
    kc = torch.full((3, 2, 16, 128), float("nan"), device=DEV).to(torch.bfloat16)
    lens = torch.zeros(3, dtype=torch.int32, device=DEV)
    out = dsa.gqa_decode_attn(q, kc, kc.clone(), lens, max_len=0)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


# ------------------------------------------------------ the whole step ---
def _step(cfg, inp, num_parts=0, inv_freq=None, scale=0.0):
    d = dev(inp)
    max_len = int(inp["lens"].max())
    B, Hq, D = d["q"].shape
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len, num_parts)
    st = {"y": torch.empty_like(d["x"]), "residual": d["residual"].clone(), "q": d["q"].clone(),
          "k_cache": d["k_cache"], "v_cache": d["v_cache"], "out": torch.empty_like(d["q"])}
    dsa.decode_step(d["x"], st["residual"], d["norm_w"], st["y"], st["q"], d["k_new"], d["v_new"],
                    st["k_cache"], st["v_cache"], d["pos"], d["lens"], st["out"], ws,
                    theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                    k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len, num_parts=num_parts,
                    inv_freq=inv_freq, scale=scale)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    return st


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_step_staged(name):
    """dec_decode_step; each stage against the oracle on that stage's own inputs."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    st = _step(cfg, inp)
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]), cfg.eps)
    check_float(f64(st["y"]), y_ref, "y")
    check_ulp(f64(st["residual"]), s_ref, "residual")
    pos = inp["pos"].numpy()
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    q_ref = O.qknorm_rope(f64(inp["q"]), qn, pos, cfg.theta, cfg.layout, cfg.eps)
    check_float(f64(st["q"]), q_ref, "q")
    lens = inp["lens"].numpy()
    out_ref = O.gqa_decode_attention(f64(st["q"]), f64(st["k_cache"]), f64(st["v_cache"]), lens)
    check_float(f64(st["out"]), out_ref, "out")


@pytest.mark.parametrize("name", ["tiny", "serving_small"])
def test_step_graph_matches_eager(name):
    """The captured step replays the same kernels: same bits as the eager call."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    eager = _step(cfg, inp)
    d = dev(inp)
    max_len = int(inp["lens"].max())
    B, Hq, D = d["q"].shape
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    buf = {"y": torch.empty_like(d["x"]), "residual": d["residual"].clone(), "q": d["q"].clone(),
           "out": torch.empty_like(d["q"])}
    kw = dict(x=d["x"], residual=buf["residual"], norm_w=d["norm_w"], y=buf["y"], q=buf["q"],
              k_new=d["k_new"], v_new=d["v_new"], k_cache=d["k_cache"], v_cache=d["v_cache"],
              pos=d["pos"], lens=d["lens"], out=buf["out"], workspace=ws, theta=cfg.theta,
              layout=cfg.layout, q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps,
              max_len=max_len)
    g = dsa.StepGraph(**kw)  # runs once eagerly, then captures
    buf["residual"].copy_(d["residual"])
    buf["q"].copy_(d["q"])
    g.replay()
    torch.cuda.synchronize()
    for k in ("y", "residual", "q", "out"):
        assert torch.equal(buf[k].view(torch.int16), eager[k].view(torch.int16)), k
    assert dsa.device_errors(ws) == 0


def test_step_graph_with_host_io():
    """One replay of the graph with packed host staging copies the inputs in, runs the
    step and copies the results out: the host buffers then hold what the eager call
    computes."""
    cfg = SMALL["serving_small"]
    inp = W.make_inputs(cfg)
    eager = _step(cfg, inp)
    d = dev(inp)
    max_len = int(inp["lens"].max())
    B, Hq, D = d["q"].shape
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    names_in = ["x", "q", "k_new", "v_new", "pos", "lens"]
    spec_in = [(k, tuple(inp[k].shape), inp[k].dtype) for k in names_in]
    spec_io = [("residual", tuple(inp["residual"].shape), torch.bfloat16),
               ("out", (B, Hq, D), torch.bfloat16), ("y", tuple(inp["x"].shape), torch.bfloat16)]
    n_in, n_io = dsa.packed_size(spec_in), dsa.packed_size(spec_io)
    dbuf = torch.empty(n_in + n_io, dtype=torch.uint8, device=DEV)
    hbuf = torch.empty(n_in + n_io, dtype=torch.uint8).pin_memory()
    dv, _ = dsa.packed_views(spec_in + spec_io, dbuf)
    hv, _ = dsa.packed_views(spec_in + spec_io, hbuf)
    for k in names_in + ["residual"]:
        hv[k].copy_(inp[k])
    n_up = n_in + dsa.packed_size(spec_io[:1])  # inputs and the residual go up
    g = dsa.StepGraph(copies_in=[(hbuf[:n_up], dbuf[:n_up])], copies_out=[(dbuf[n_in:], hbuf[n_in:])],
                      x=dv["x"], residual=dv["residual"], norm_w=d["norm_w"], y=dv["y"], q=dv["q"],
                      k_new=dv["k_new"], v_new=dv["v_new"], k_cache=d["k_cache"], v_cache=d["v_cache"],
                      pos=dv["pos"], lens=dv["lens"], out=dv["out"], workspace=ws, theta=cfg.theta,
                      layout=cfg.layout, q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps,
                      max_len=max_len)
    for k in names_in + ["residual"]:
        hv[k].copy_(inp[k])  # the eager warm-up inside the constructor rotated q in place
    hv["out"].zero_()
    hv["y"].zero_()
    g.replay()
    torch.cuda.synchronize()
    for k in ("out", "y", "residual"):
        assert torch.equal(hv[k].view(torch.int16), eager[k].cpu().view(torch.int16)), k


@pytest.mark.parametrize("name", ["llama3_small", "serving_small", "long_small", "tiny"])
@pytest.mark.parametrize("window", [1, 7, 64, 129, 1000, 10 ** 6])
@pytest.mark.parametrize("num_parts", [0, 3])
def test_sliding_window_attention(name, window, num_parts):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    d = dev(inp)
    lens = inp["lens"].numpy()
    max_len = int(lens.max())
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len, num_parts)
    out = dsa.gqa_decode_attn(d["q"], kc.to(DEV), vc.to(DEV), d["lens"], max_len=max_len,
                              workspace=ws, num_parts=num_parts, window=window)
    torch.cuda.synchronize()
    ref = O.gqa_decode_attention(f64(inp["q"]), f64(kc), f64(vc), lens, window=window)
    check_float(f64(out), ref, f"{name} window={window} parts={num_parts}")
    assert dsa.device_errors(ws) == 0


def _every_head_ref(q64, k_cache, v_cache, lens, G, scale, window=None):
    """The oracle's attention for every (sequence, query head), one (sequence, KV head)
    pair at a time (the pair's K and V in fp64, at most a few hundred MB)."""
    B, Hq, D = q64.shape
    Hkv = k_cache.shape[1]
    ref = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        lo = 0 if window is None else max(0, L - window)
        if L == 0:
            continue
        for g in range(Hkv):
            K = k_cache[b, g, lo:L].double().numpy()
            V = v_cache[b, g, lo:L].double().numpy()
            for hh in range(G):
                ref[b, g * G + hh] = O.attend_one(q64[b, g * G + hh], K, V, scale)
    return ref


def _full_step(cfg, inp, window=0):
    """The decode step on a full workload in the benchmark's launch configuration
    (num_parts = 0: one CTA per SM, or the one-launch kernel on short contexts), with
    guard copies of the caches to check every slot but the appended one."""
    d = dev(inp)
    max_len = int(inp["lens"].max())
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    kc0, vc0 = d["k_cache"].clone(), d["v_cache"].clone()
    st = {"y": torch.empty_like(d["x"]), "residual": d["residual"].clone(), "q": d["q"].clone(),
          "out": torch.empty_like(d["q"])}
    dsa.decode_step(d["x"], st["residual"], d["norm_w"], st["y"], st["q"], d["k_new"], d["v_new"],
                    d["k_cache"], d["v_cache"], d["pos"], d["lens"], st["out"], ws,
                    theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                    k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len, window=window)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    # every slot but pos[b] is untouched (compared on the device, bit for bit)
    pos_d = d["pos"].long()
    bidx = torch.arange(cfg.B, device=DEV)
    for c, c0 in ((d["k_cache"], kc0), (d["v_cache"], vc0)):
        same = (c.view(torch.int16) == c0.view(torch.int16)).all(dim=-1)  # [B, Hkv, T]
        same[bidx, :, pos_d] = True
        assert bool(same.all()), "a cache slot other than pos[b] changed"
    del kc0, vc0
    st["k_cache"], st["v_cache"] = d["k_cache"].cpu(), d["v_cache"].cpu()
    return st


@pytest.mark.parametrize("name,window", [("long_context_131k", 4096), ("serving_mix", 1024)])
def test_sliding_window_full_size_every_head(name, window):
    """A windowed step at full size: every head of the output against the oracle."""
    cfg = W.CONFIGS[name]
    inp = W.make_inputs(cfg)
    st = _full_step(cfg, inp, window=window)
    lens = inp["lens"].numpy()
    ref = _every_head_ref(f64(st["q"]), st["k_cache"], st["v_cache"], lens, cfg.G,
                          1.0 / math.sqrt(cfg.D), window=window)
    check_float(f64(st["out"]), ref, f"{name} window {window}, every head")


FULL = ["qwen3_0p6b_ctx512", "llama3_8b_batched", "long_context_131k", "serving_mix"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_head(name):
    """The full workload in the benchmark's launch configuration, every output element
    against the oracle: y and the residual, the rotated q, the appended K and V slots,
    every other cache slot unchanged, and every (sequence, query head) of the output."""
    cfg = W.CONFIGS[name]
    inp = W.make_inputs(cfg)
    st = _full_step(cfg, inp)
    lens = inp["lens"].numpy()
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]), cfg.eps)
    check_float(f64(st["y"]), y_ref, f"{name} y")
    check_ulp(f64(st["residual"]), s_ref, f"{name} residual")
    pos = inp["pos"].numpy()
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    kn = None if inp["k_norm_w"] is None else f64(inp["k_norm_w"])
    q_ref = O.qknorm_rope(f64(inp["q"]), qn, pos, cfg.theta, cfg.layout, cfg.eps)
    check_float(f64(st["q"]), q_ref, f"{name} q")
    k_ref = O.qknorm_rope(f64(inp["k_new"]), kn, pos, cfg.theta, cfg.layout, cfg.eps)
    bidx = np.arange(cfg.B)
    check_ulp(f64(st["k_cache"][bidx, :, pos]), k_ref, f"{name} appended K")
    assert torch.equal(st["v_cache"][bidx, :, pos].view(torch.int16),
                       inp["v_new"].view(torch.int16)), "the V slot is not a bit copy"
    ref = _every_head_ref(f64(st["q"]), st["k_cache"], st["v_cache"], lens, cfg.G,
                          1.0 / math.sqrt(cfg.D))
    check_float(f64(st["out"]), ref, f"{name} every head")


def test_split_partials_full_size_131k():
    """Every partial of the split pass on the 131072-token context at the benchmark's
    split (one CTA per SM) against the oracle's partial over the same token range."""
    cfg = W.LONG_CONTEXT
    inp = W.make_inputs(cfg)
    kc, vc = with_new_token(inp)
    d = dev(inp)
    lens = inp["lens"].numpy()
    B, Hq, Hkv, D, G = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.G
    max_len = int(lens.max())
    parts = dsa.default_parts(B, Hkv, D, max_len)
    assert parts == torch.cuda.get_device_properties(0).multi_processor_count
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, max_len, parts)
    dsa.gqa_decode_split(d["q"], kc.to(DEV), vc.to(DEV), d["lens"], ws, max_len=max_len,
                         num_parts=parts)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    slots = _slots(B, Hkv, parts)
    body = ws[dsa.WORKSPACE_HEADER_BYTES:].view(torch.float32).cpu().numpy()
    o_ws = body[:slots * G * D].reshape(slots, G, D)
    lse_ws = body[slots * G * D: slots * G * D + slots * G].reshape(slots, G)
    qf = f64(inp["q"])
    scale = 1.0 / math.sqrt(D)
    got, want, n = [], [], 0
    for (b, g), lst in _partition(lens, Hkv, parts).items():
        K, V = kc[b, g].double().numpy(), vc[b, g].double().numpy()
        for (c, t0, t1) in lst:
            slot = c + b * Hkv + g
            for hh in range(G):
                o_ref, lse_ref = O.attention_partial(qf[b, g * G + hh], K[t0:t1], V[t0:t1], scale)
                got.append(o_ws[slot, hh])
                want.append(o_ref)
                assert abs(lse_ws[slot, hh] * LN2 - lse_ref) <= 1e-4 * max(1.0, abs(lse_ref)), \
                    (b, g, c, hh)
                n += 1
    assert n >= 5 * parts  # every piece of every pair
    check_float(np.array(got), np.array(want), "131k partials", abs_tol=1e-3, rel_rms=1e-4)


# ------------------------------------------------- one-launch step (short contexts)
ONE_LAUNCH = ["tiny", "qwen3_ctx128", "qwen3_ctx512", "llama3_small"]


def test_one_launch_is_chosen_for_short_contexts():
    for name in ONE_LAUNCH:
        cfg = SMALL[name]
        max_len = int(W.make_inputs(cfg, with_cache=False)["lens"].max())
        assert dsa.decode_step_launches(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len) == 1, name
    for name in ("serving_small", "long_small"):
        cfg = SMALL[name]
        max_len = int(W.make_inputs(cfg, with_cache=False)["lens"].max())
        assert dsa.decode_step_path(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len) == dsa.STEP_STREAM, name
        assert dsa.decode_step_launches(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len) == 2, name


@pytest.mark.parametrize("name", ONE_LAUNCH)
def test_one_launch_matches_separate_calls(name):
    """The one-launch step against K1, K2 and the attention called one by one: y, the
    residual, the rotated q, both caches and the output bit for bit (the attention call
    takes the same one-launch kernel for these shapes), and the output within the
    oracle's tolerance."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    st = _step(cfg, inp)
    d = dev(inp)
    max_len = int(inp["lens"].max())
    r2, q2 = d["residual"].clone(), d["q"].clone()
    kc2, vc2 = d["k_cache"].clone(), d["v_cache"].clone()
    y2 = dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=r2, eps=cfg.eps)
    dsa.qknorm_rope_kv_append(q2, d["k_new"], d["v_new"], kc2, vc2, d["pos"], cfg.theta,
                              cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps)
    out2 = dsa.gqa_decode_attn(q2, kc2, vc2, d["lens"], max_len=max_len)
    torch.cuda.synchronize()
    for k, a, b in (("y", st["y"], y2), ("residual", st["residual"], r2), ("q", st["q"], q2),
                    ("k_cache", st["k_cache"], kc2), ("v_cache", st["v_cache"], vc2),
                    ("out", st["out"], out2)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), k
    ref = O.gqa_decode_attention(f64(q2), f64(kc2), f64(vc2), inp["lens"].numpy())
    check_float(f64(st["out"]), ref, "one launch")
    # the split pass and its merge, forced by an explicit split count, on the same inputs
    out3 = dsa.gqa_decode_attn(q2, kc2, vc2, d["lens"], max_len=max_len,
                               num_parts=dsa.default_parts(cfg.B, cfg.Hkv, cfg.D, max_len))
    torch.cuda.synchronize()
    check_float(f64(out3), ref, "split pass + merge")


STREAMING = {
    "llama3_small": SMALL["llama3_small"],
    "long_small": SMALL["long_small"],
    "serving_small": SMALL["serving_small"],
    # 152 split CTAs of 267 rows: pair (9, 1)'s new slot (row 1499) is a run of its own,
    # and the run before it ends one row short, so its last tile loads the slot that
    # another CTA is writing in the same launch
    "serving_slot_at_piece_edge": W.small_variant(W.SERVING_MIX, B=24, max_len=1500),
}


@pytest.mark.parametrize("name", list(STREAMING))
@pytest.mark.parametrize("window", [0, 333])
def test_streaming_step_matches_separate_calls(name, window):
    """The streaming form of the step (the fused RMSNorm + rotation launch, then the split
    pass and its merge in one cooperative launch) against K1, K2 and the attention called
    one by one: the residual, the rotated q, both caches and the output bit for bit (the
    same rotation code and the same split-pass arithmetic), y within one ulp, and every
    stage against the oracle. The last case puts a sequence's new slot in a run of its
    own, right after another CTA's run that reads it as padding."""
    cfg = STREAMING[name]
    inp = W.make_inputs(cfg)
    d = dev(inp)
    max_len = int(inp["lens"].max())
    B, Hq, D = d["q"].shape
    if dsa.decode_step_path(B, Hq, cfg.Hkv, D, max_len, window) != dsa.STEP_STREAM:
        pytest.skip("this device runs the shape in three launches")
    ws = dsa.alloc_workspace(B, Hq, cfg.Hkv, D, max_len)
    st = {"y": torch.empty_like(d["x"]), "residual": d["residual"].clone(), "q": d["q"].clone(),
          "k_cache": d["k_cache"].clone(), "v_cache": d["v_cache"].clone(),
          "out": torch.empty_like(d["q"])}
    dsa.decode_step(d["x"], st["residual"], d["norm_w"], st["y"], st["q"], d["k_new"],
                    d["v_new"], st["k_cache"], st["v_cache"], d["pos"], d["lens"], st["out"], ws,
                    theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                    k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len, window=window)
    r2, q2 = d["residual"].clone(), d["q"].clone()
    kc2, vc2 = d["k_cache"].clone(), d["v_cache"].clone()
    y2 = dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=r2, eps=cfg.eps)
    dsa.qknorm_rope_kv_append(q2, d["k_new"], d["v_new"], kc2, vc2, d["pos"], cfg.theta,
                              cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps)
    out2 = dsa.gqa_decode_attn(q2, kc2, vc2, d["lens"], max_len=max_len, window=window)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    for k, a, b in (("residual", st["residual"], r2), ("q", st["q"], q2),
                    ("k_cache", st["k_cache"], kc2), ("v_cache", st["v_cache"], vc2),
                    ("out", st["out"], out2)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), k
    check_ulp(f64(st["y"]), f64(y2), "y against the standalone RMSNorm")
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]),
                                      cfg.eps)
    check_float(f64(st["y"]), y_ref, "y")
    check_ulp(f64(st["residual"]), s_ref, "residual")
    ref = O.gqa_decode_attention(f64(st["q"]), f64(st["k_cache"]), f64(st["v_cache"]),
                                 inp["lens"].numpy(), window=window if window else None)
    check_float(f64(st["out"]), ref, "out")


@pytest.mark.parametrize("name", ONE_LAUNCH)
@pytest.mark.parametrize("window", [0, 1, 37, 4096])
def test_attention_call_one_launch(name, window):
    """The attention call alone on a short context (one launch): against the oracle,
    with host-visible error bits for clamped lengths, an empty sequence giving zeros,
    and the inputs left untouched."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    d = dev(inp)
    kc, vc = with_new_token(inp)
    kc, vc = kc.to(DEV), vc.to(DEV)
    lens = inp["lens"].clone()
    lens[-1] = 0
    max_len = int(inp["lens"].max())
    assert dsa.decode_step_launches(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len, window) == 1
    q0, k0, v0 = d["q"].clone(), kc.clone(), vc.clone()
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    out = torch.full_like(d["q"], 3.0)
    if window:
        dsa.gqa_decode_attn(d["q"], kc, vc, lens.to(DEV), max_len=max_len, workspace=ws, out=out,
                            window=window)
    else:
        dsa.gqa_decode_attn(d["q"], kc, vc, lens.to(DEV), max_len=max_len, workspace=ws, out=out)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    ref = O.gqa_decode_attention(f64(d["q"]), f64(kc), f64(vc), lens.numpy(),
                                 window=window or None)
    check_float(f64(out), ref, f"{name} window {window}")
    assert torch.equal(out[-1], torch.zeros_like(out[-1]))
    for a, b in ((d["q"], q0), (kc, k0), (vc, v0)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "qwen3_ctx512", "llama3_small"])
@pytest.mark.parametrize("window", [1, 5, 64, 300, 4096])
def test_one_launch_window(name, window):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    d = dev(inp)
    max_len = int(inp["lens"].max())
    assert dsa.decode_step_launches(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len, window) == 1
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    y, out = torch.empty_like(d["x"]), torch.empty_like(d["q"])
    resid, q = d["residual"].clone(), d["q"].clone()
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    dsa.decode_step(d["x"], resid, d["norm_w"], y, q, d["k_new"], d["v_new"], kc, vc, d["pos"],
                    d["lens"], out, ws, theta=cfg.theta, layout=cfg.layout,
                    q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len,
                    window=window)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    ref = O.gqa_decode_attention(f64(q), f64(kc), f64(vc), inp["lens"].numpy(), window=window)
    check_float(f64(out), ref, f"{name} window {window}")


def test_one_launch_edge_cases():
    """A position outside the cache (the sequence is skipped: q as given, no append, the
    flag raised), a length beyond T_cap (clamped, flagged) and an empty sequence (zeros),
    each as the three-launch path treats them."""
    cfg = W.small_variant(W.QWEN3_512, B=4, max_len=200)
    inp = W.make_inputs(cfg)
    T_cap = inp["t_cap"]
    pos = inp["pos"].clone()
    lens = inp["lens"].clone()
    pos[1] = T_cap + 3          # skipped (its slot would have been lens - 1: attend below it)
    lens[1] = max(int(lens[1]) - 1, 0)
    lens[2] = T_cap + 50        # clamped to T_cap
    lens[3] = 0                 # empty
    d = dev(inp)
    d["pos"], d["lens"] = pos.to(DEV), lens.to(DEV)
    max_len = T_cap
    assert dsa.decode_step_launches(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len) == 1
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    y, out = torch.empty_like(d["x"]), torch.full_like(d["q"], 7.0)
    resid, q = d["residual"].clone(), d["q"].clone()
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    dsa.decode_step(d["x"], resid, d["norm_w"], y, q, d["k_new"], d["v_new"], kc, vc, d["pos"],
                    d["lens"], out, ws, theta=cfg.theta, layout=cfg.layout,
                    q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len)
    torch.cuda.synchronize()
    err = dsa.device_errors(ws)
    assert err & dsa.DEVERR_POS_SKIPPED and err & dsa.DEVERR_LEN_CLAMPED
    assert torch.equal(q[1].view(torch.int16), d["q"][1].view(torch.int16))  # not rotated
    assert torch.equal(kc[1].view(torch.int16), d["k_cache"][1].view(torch.int16))  # no append
    assert torch.equal(out[3], torch.zeros_like(out[3]))
    eff = np.minimum(np.maximum(lens.numpy(), 0), T_cap)
    ref = O.gqa_decode_attention(f64(q), f64(kc), f64(vc), eff)
    # the clamped sequence attends to every slot, NaN sentinels included: compare the rest
    for b in (0, 1, 3):
        check_float(f64(out[b]), ref[b], f"sequence {b}")


# ----------------------------------------- RoPE frequency tables (context extension)
def _tables(D, theta, scaling, factor, seed=0):
    """(the GPU's table, the oracle's): the library's builder and the oracle's, each
    on its own side; a "custom" table is a seeded input given to both."""
    if scaling == "custom":
        rng = np.random.default_rng(seed)
        t = rng.uniform(0.0, 1.0, D // 2)
        t[0], t[-1] = 1.0, 0.0  # the ends of the allowed range
        return torch.tensor(t, dtype=torch.float64), t
    return (dsa.rope_inv_freq(D, theta, scaling, factor),
            O.rope_scaled_inv_freq(D, np.float32(theta), scaling, factor))


@pytest.mark.parametrize("scaling,factor", [("linear", 4.0), ("ntk", 8.0), ("custom", 0.0)])
@pytest.mark.parametrize("layout", ["neox", "interleaved"])
@pytest.mark.parametrize("D", [64, 128])
def test_append_rope_tables(scaling, factor, layout, D):
    """K2 with a context-extension table, at positions up to 131071."""
    cfg = W.BlockConfig("append_tables", B=5, hidden=256, Hq=8, Hkv=2, D=D, theta=5e5,
                        layout=layout, qk_norm=True, lens_kind="list",
                        lens_args=(1, 2, 900, 131072, 77777), t_cap=131072, seed=4)
    inp = W.make_inputs(cfg, with_cache=False)
    T = 131072
    inp["k_cache"] = W.nan_bf16((cfg.B, cfg.Hkv, T, D))
    inp["v_cache"] = W.nan_bf16((cfg.B, cfg.Hkv, T, D))
    _append_check(cfg, inp, f"{scaling}/{layout}/{D}", _tables(D, cfg.theta, scaling, factor))


@pytest.mark.parametrize("name", ["tiny", "qwen3_ctx512", "llama3_small", "serving_small",
                                  "long_small"])
@pytest.mark.parametrize("scaling,factor", [("linear", 8.0), ("ntk", 4.0)])
def test_decode_step_rope_tables(name, scaling, factor):
    """The whole step (one launch for the short contexts, three for the rest) with a
    scaled table: the rotated q and the appended K against the oracle with its own
    table, the output against the oracle's attention over the GPU's caches."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    gpu_t, ref_t = _tables(cfg.D, cfg.theta, scaling, factor)
    st = _step(cfg, inp, inv_freq=gpu_t)
    pos = inp["pos"].numpy()
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    kn = None if inp["k_norm_w"] is None else f64(inp["k_norm_w"])
    check_float(f64(st["q"]), O.qknorm_rope(f64(inp["q"]), qn, pos, cfg.theta, cfg.layout,
                                            cfg.eps, ref_t), "q")
    k_rot = O.qknorm_rope(f64(inp["k_new"]), kn, pos, cfg.theta, cfg.layout, cfg.eps, ref_t)
    new_k = np.stack([f64(st["k_cache"][b, :, int(pos[b])]) for b in range(cfg.B)])
    check_ulp(new_k, k_rot, "appended k", ulps=1.0)
    out_ref = O.gqa_decode_attention(f64(st["q"]), f64(st["k_cache"]), f64(st["v_cache"]),
                                     inp["lens"].numpy())
    check_float(f64(st["out"]), out_ref, "out")


@pytest.mark.parametrize("name", ["tiny", "llama3_small", "serving_small"])
def test_unscaled_table_is_the_default(name):
    """The builder's unscaled table given explicitly: the same bits as no table."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    a = _step(cfg, inp)
    b = _step(cfg, inp, inv_freq=dsa.rope_inv_freq(cfg.D, cfg.theta))
    for k in ("q", "k_cache", "out"):
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k


def test_rope_table_rejects():
    """Tables outside [0, 1], not finite, or in device memory are refused before any
    launch, and the inputs are left as they were."""
    import ctypes
    cfg = SMALL["qwen3_ctx128"]
    inp = W.make_inputs(cfg)
    d = dev(inp)
    q = d["q"].clone()
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    good = dsa.rope_inv_freq(cfg.D, cfg.theta)
    for bad_value in (1.5, -0.25, float("nan"), float("inf")):
        t = good.clone()
        t[5] = bad_value
        with pytest.raises(dsa.DecAttnError) as e:
            dsa.qknorm_rope_kv_append(q, d["k_new"], d["v_new"], kc, vc, d["pos"], cfg.theta,
                                      cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps,
                                      inv_freq=t)
        assert e.value.status == 1 and "inv_freq" in str(e.value)
    on_device = good.to(DEV)
    L = dsa.lib()
    B, Hq, D = q.shape
    st = L.dec_qknorm_rope_kv_append(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(d["k_new"].data_ptr()),
        ctypes.c_void_p(d["v_new"].data_ptr()), ctypes.c_void_p(d["q_norm_w"].data_ptr()),
        ctypes.c_void_p(d["k_norm_w"].data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(d["pos"].data_ptr()), B, Hq, cfg.Hkv, D,
        kc.shape[2], cfg.theta, 0, ctypes.c_void_p(on_device.data_ptr()), cfg.eps, None, None)
    assert st == 1 and b"host memory" in L.dec_last_error()
    with pytest.raises(ValueError):
        dsa.qknorm_rope_kv_append(q, d["k_new"], d["v_new"], kc, vc, d["pos"], cfg.theta,
                                  cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps,
                                  inv_freq=on_device)
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.int16), d["q"].view(torch.int16))
    assert torch.equal(kc.view(torch.int16), d["k_cache"].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "qwen3_ctx512", "llama3_small", "serving_small",
                                  "long_small"])
def test_decode_step_yarn(name):
    """YaRN: the step with the library's YaRN table and the softmax scale that carries the
    method's temperature, against the oracle's form of the method (rotated q and k both
    multiplied by 0.1 ln(s) + 1, softmax scale 1/sqrt(D)): the rotation against the
    oracle's own table, the output against the oracle's attention over the GPU's rotated
    q and caches with that multiplier applied."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    s, ctx = 8.0, 256
    t_gpu = dsa.rope_inv_freq(cfg.D, cfg.theta, "yarn", s, ctx)
    t_ref = O.rope_scaled_inv_freq(cfg.D, np.float32(cfg.theta), "yarn", s, ctx)
    st = _step(cfg, inp, inv_freq=t_gpu, scale=dsa.yarn_softmax_scale(cfg.D, s))
    pos = inp["pos"].numpy()
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    kn = None if inp["k_norm_w"] is None else f64(inp["k_norm_w"])
    check_float(f64(st["q"]), O.qknorm_rope(f64(inp["q"]), qn, pos, cfg.theta, cfg.layout,
                                            cfg.eps, t_ref), "q")
    k_rot = O.qknorm_rope(f64(inp["k_new"]), kn, pos, cfg.theta, cfg.layout, cfg.eps, t_ref)
    new_k = np.stack([f64(st["k_cache"][b, :, int(pos[b])]) for b in range(cfg.B)])
    check_ulp(new_k, k_rot, "appended k", ulps=1.0)
    m = O.yarn_attention_factor(s)
    out_ref = O.gqa_decode_attention(m * f64(st["q"]), m * f64(st["k_cache"]),
                                     f64(st["v_cache"]), inp["lens"].numpy())
    check_float(f64(st["out"]), out_ref, "out")


@pytest.mark.parametrize("name", ["qwen3_ctx512", "serving_small", "long_small"])
@pytest.mark.parametrize("window", [33, 400])
def test_decode_step_rope_table_with_window(name, window):
    """A context-extension table and a sliding window in the same step (one launch for
    the Qwen3-shaped case, three for the others)."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg)
    gpu_t, ref_t = _tables(cfg.D, cfg.theta, "ntk", 4.0)
    d = dev(inp)
    max_len = int(inp["lens"].max())
    ws = dsa.alloc_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    y, out = torch.empty_like(d["x"]), torch.empty_like(d["q"])
    resid, q = d["residual"].clone(), d["q"].clone()
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    dsa.decode_step(d["x"], resid, d["norm_w"], y, q, d["k_new"], d["v_new"], kc, vc, d["pos"],
                    d["lens"], out, ws, theta=cfg.theta, layout=cfg.layout,
                    q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len,
                    window=window, inv_freq=gpu_t)
    torch.cuda.synchronize()
    assert dsa.device_errors(ws) == 0
    pos = inp["pos"].numpy()
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    check_float(f64(q), O.qknorm_rope(f64(inp["q"]), qn, pos, cfg.theta, cfg.layout, cfg.eps,
                                      ref_t), "q")
    ref = O.gqa_decode_attention(f64(q), f64(kc), f64(vc), inp["lens"].numpy(), window=window)
    check_float(f64(out), ref, f"{name} window {window}")
