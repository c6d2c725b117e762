"""Guard words around every buffer a decode step writes (GPU only).

Each output (y, the residual, q, out, both caches and the workspace) is a view into a
larger buffer whose bytes just before and after the view hold a fixed pattern; after
the step, on the one-launch and the three-launch paths, with and without a sliding
window, every guard byte must still hold it. A kernel that stores one element past an
edge of its tensor fails here even when its results are right.
"""
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 4096  # bytes on each side (16-byte aligned views, so the alignment rules hold)
PATTERN = 0xA5


def _guarded(t: torch.Tensor):
    """A device copy of t inside a buffer with GUARD pattern bytes on each side."""
    n = t.numel() * t.element_size()
    buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
    view = buf[GUARD:GUARD + n].view(t.dtype).view(t.shape)
    view.copy_(t.to(DEV))
    return buf, view


def _intact(buf) -> bool:
    return bool((buf[:GUARD] == PATTERN).all()) and bool((buf[-GUARD:] == PATTERN).all())


CASES = {
    "tiny_one_launch": (W.TINY, 0),
    "qwen_one_launch": (W.QWEN3_512, 0),
    "serving_three_launch": (W.small_variant(W.SERVING_MIX, B=24, max_len=1500), 0),
    "llama_three_launch_window": (W.small_variant(W.LLAMA3_BATCHED, B=4, max_len=3000), 700),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_step_writes_nothing_outside_its_buffers(name):
    cfg, window = CASES[name]
    inp = W.make_inputs(cfg)
    max_len = int(inp["lens"].max())
    g = {}
    for k in ("x", "residual", "norm_w", "q", "k_new", "v_new", "k_cache", "v_cache", "pos", "lens"):
        g[k] = _guarded(inp[k])
    g["y"] = _guarded(torch.zeros_like(inp["x"]))
    g["out"] = _guarded(torch.zeros_like(inp["q"]))
    ws_bytes = dsa.attn_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    g["ws"] = _guarded(torch.zeros(ws_bytes, dtype=torch.uint8))
    qn = inp["q_norm_w"].to(DEV) if cfg.qk_norm else None
    kn = inp["k_norm_w"].to(DEV) if cfg.qk_norm else None
    v = {k: b[1] for k, b in g.items()}
    dsa.decode_step(v["x"], v["residual"], v["norm_w"], v["y"], v["q"], v["k_new"], v["v_new"],
                    v["k_cache"], v["v_cache"], v["pos"], v["lens"], v["out"], v["ws"],
                    theta=cfg.theta, layout=cfg.layout, q_norm_w=qn, k_norm_w=kn, eps=cfg.eps,
                    max_len=max_len, window=window)
    torch.cuda.synchronize()
    assert dsa.device_errors(v["ws"]) == 0
    assert torch.isfinite(v["out"].float()).all()
    for k, (buf, _) in g.items():
        assert _intact(buf), f"{name}: a guard byte next to {k} changed"


def test_attention_call_and_sublayer_guards():
    """The split pass and merge called on their own, and the attention sublayer."""
    cfg = W.small_variant(W.SERVING_MIX, B=24, max_len=1500, seed=3)
    inp = W.make_inputs(cfg)
    max_len = int(inp["lens"].max())
    g = {k: _guarded(inp[k]) for k in ("q", "k_cache", "v_cache", "lens")}
    parts = 37
    ws_bytes = dsa.attn_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len, parts)
    g["ws"] = _guarded(torch.zeros(ws_bytes, dtype=torch.uint8))
    g["out"] = _guarded(torch.zeros_like(inp["q"]))
    v = {k: b[1] for k, b in g.items()}
    dsa.gqa_decode_split(v["q"], v["k_cache"], v["v_cache"], v["lens"], v["ws"], max_len=max_len,
                         num_parts=parts)
    dsa.split_merge(v["ws"], v["lens"], v["out"], cfg.Hkv, inp["t_cap"], max_len=max_len,
                    num_parts=parts)
    torch.cuda.synchronize()
    for k, (buf, _) in g.items():
        assert _intact(buf), f"split/merge: a guard byte next to {k} changed"

    wts = W.make_projection_weights(cfg)
    s = {k: _guarded(inp[k]) for k in ("x", "residual", "norm_w", "k_cache", "v_cache", "pos",
                                       "lens", "q_norm_w", "k_norm_w")}
    s["w_qkv"] = _guarded(wts["w_qkv"])
    s["w_o"] = _guarded(wts["w_o"])
    s["out"] = _guarded(torch.zeros_like(inp["x"]))
    sb = dsa.sublayer_workspace_bytes(cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D, max_len)
    s["ws"] = _guarded(torch.zeros(sb, dtype=torch.uint8))
    u = {k: b[1] for k, b in s.items()}
    dsa.attn_sublayer(u["x"], u["residual"], u["norm_w"], u["w_qkv"], u["w_o"], u["k_cache"],
                      u["v_cache"], u["pos"], u["lens"], u["out"], u["ws"], theta=cfg.theta,
                      layout=cfg.layout, q_norm_w=u["q_norm_w"], k_norm_w=u["k_norm_w"],
                      eps=cfg.eps, max_len=max_len)
    torch.cuda.synchronize()
    for k, (buf, _) in s.items():
        assert _intact(buf), f"sublayer: a guard byte next to {k} changed"
