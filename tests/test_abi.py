"""The C ABI without a GPU: the library loads, exports every symbol that
include/decattn.h declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import decode_step_attention_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decattn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(dsa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return dsa.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 11, names
    for n in names:
        assert hasattr(L, n), f"{n} is declared in decattn.h but not exported"
    assert set(names) == set(dsa.EXPORTS), "binding and header disagree"


def test_status_strings(L):
    assert L.dec_status_string(0) == b"ok"
    assert L.dec_status_string(3) == b"workspace too small"
    assert L.dec_version() == 100


def _st(L, name, *args):
    st = getattr(L, name)(*args)
    return st, L.dec_last_error().decode()


P = ctypes.c_void_p(16 * 1024)  # a 16-byte aligned dummy address; never dereferenced


def test_rmsnorm_rejects(L):
    st, msg = _st(L, "dec_rmsnorm_residual", P, None, P, P, -1, 256, 1e-6, None)
    assert st == 1 and "B" in msg
    st, _ = _st(L, "dec_rmsnorm_residual", P, None, P, P, 2, 100, 1e-6, None)
    assert st == 2
    st, _ = _st(L, "dec_rmsnorm_residual", P, None, P, P, 2, 256, -1.0, None)
    assert st == 1
    st, _ = _st(L, "dec_rmsnorm_residual", None, None, P, P, 2, 256, 1e-6, None)
    assert st == 1
    st, msg = _st(L, "dec_rmsnorm_residual", ctypes.c_void_p(16 * 1024 + 2), None, P,
                  ctypes.c_void_p(32 * 1024), 2, 256, 1e-6, None)
    assert st == 1 and "aligned" in msg
    st, msg = _st(L, "dec_rmsnorm_residual", P, None, P, P, 2, 256, 1e-6, None)
    assert st == 1 and "alias" in msg
    st, _ = _st(L, "dec_rmsnorm_residual", None, None, None, None, 0, 256, 1e-6, None)
    assert st == 0  # B == 0 is a no-op


def test_append_out_rejects_partial_overlap(L):
    kc, vc = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20)
    q_in, q_out = ctypes.c_void_p(3 << 20), ctypes.c_void_p((3 << 20) + 256)
    st, msg = _st(L, "dec_qknorm_rope_kv_append_out", q_in, q_out, P, P, None, None, kc, vc, P,
                  2, 8, 2, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 1 and "overlap" in msg
    st, msg = _st(L, "dec_qknorm_rope_kv_append_out", None, q_out, P, P, None, None, kc, vc, P,
                  2, 8, 2, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 1 and "non-null" in msg
    st, _ = _st(L, "dec_qknorm_rope_kv_append_out", None, None, None, None, None, None, None,
                None, None, 0, 8, 2, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 0  # B == 0 is a no-op


def test_append_rejects(L):
    args = [P, P, P, None, None, P, ctypes.c_void_p(64 * 1024), P]
    st, _ = _st(L, "dec_qknorm_rope_kv_append", *args, 2, 8, 3, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 1  # Hq % Hkv
    st, _ = _st(L, "dec_qknorm_rope_kv_append", *args, 2, 8, 2, 96, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 2  # head_dim
    st, _ = _st(L, "dec_qknorm_rope_kv_append", *args, 2, 8, 2, 128, 16, -1.0, 0, None, 1e-6, None, None)
    assert st == 1  # theta
    st, _ = _st(L, "dec_qknorm_rope_kv_append", *args, 2, 8, 2, 128, 16, 1e4, 7, None, 1e-6, None, None)
    assert st == 1  # layout
    a2 = [P, P, P, P, None, P, ctypes.c_void_p(64 * 1024), P]
    st, msg = _st(L, "dec_qknorm_rope_kv_append", *a2, 2, 8, 2, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 1 and "both" in msg


def test_attention_rejects(L):
    # explicit num_parts, so no device query happens
    base = [P, P, ctypes.c_void_p(64 * 1024), P]
    st, _ = _st(L, "dec_gqa_decode_split", *base, 2, 12, 8, 128, 64, 64, 0.0, 4, P, 1 << 20, None)
    assert st == 1  # Hq % Hkv
    st, _ = _st(L, "dec_gqa_decode_split", *base, 2, 32, 2, 128, 64, 64, 0.0, 4, P, 1 << 20, None)
    assert st == 2  # group of 16 heads
    st, _ = _st(L, "dec_gqa_decode_split", *base, 2, 8, 2, 80, 64, 64, 0.0, 4, P, 1 << 20, None)
    assert st == 2  # head_dim
    st, _ = _st(L, "dec_gqa_decode_split", *base, 2, 8, 2, 128, 64, 65, 0.0, 4, P, 1 << 20, None)
    assert st == 1  # max_len > T_cap
    st, _ = _st(L, "dec_gqa_decode_split", *base, 2, 8, 2, 128, 64, 64, 0.0, 4, None, 1 << 20, None)
    assert st == 3  # no workspace
    need = L.dec_attn_workspace_bytes(2, 8, 2, 128, 64, 4)
    st, msg = _st(L, "dec_gqa_decode_split", *base, 2, 8, 2, 128, 64, 64, 0.0, 4, P, need - 256, None)
    assert st == 3 and "needed" in msg
    st, _ = _st(L, "dec_gqa_decode_split", *base, 2, 8, 2, 128, 64, 64, float("nan"), 4, P, need, None)
    assert st == 1
    st, _ = _st(L, "dec_gqa_decode_split", *base, 9000, 8, 2, 128, 64, 64, 0.0, 4, P, 1 << 30, None)
    assert st == 2  # batch beyond the split pass's prefix buffer
    st, _ = _st(L, "dec_split_merge", P, 1 << 20, P, P, 2, 8, 2, 128, 64, 64, -1, None)
    assert st == 1
    st, _ = _st(L, "dec_gqa_decode_attn", *base, None, 0, 8, 2, 128, 64, 64, 0.0, 4, None, 0, None)
    assert st == 0  # B == 0 is a no-op


def test_window_rejects(L):
    base = [P, P, ctypes.c_void_p(64 * 1024), P, ctypes.c_void_p(128 * 1024)]
    st, msg = _st(L, "dec_gqa_decode_attn_window", *base, 2, 8, 2, 128, 64, 64, 0, 0.0, 4, P,
                  1 << 20, None)
    assert st == 1 and "window" in msg


def test_decode_step_launch_rule(L):
    """Which path dec_decode_step takes (pure host logic): one launch for at most 1024
    attended rows, at most 64 (sequence, KV head) pairs and at most 8 query heads per KV
    head; else two where the device runs the attention as one cooperative launch, and
    three here, with no device to ask."""
    f = L.dec_decode_step_launches
    assert f(1, 4, 1, 64, 128, 0) == 1          # tiny
    assert f(1, 16, 8, 128, 512, 0) == 1        # Qwen3-shaped ctx 512
    assert f(1, 16, 8, 128, 1024, 0) == 1
    assert f(1, 16, 8, 128, 1025, 0) == 3       # too many rows
    assert f(1, 32, 8, 128, 131072, 1000) == 1  # a window bounds the rows attended
    assert f(8, 64, 8, 128, 512, 0) == 1        # 64 pairs
    assert f(9, 64, 8, 128, 512, 0) == 3        # 72 pairs
    assert f(1, 16, 1, 128, 128, 0) == 3        # 16 query heads per KV head
    assert f(1, 4, 1, 96, 128, 0) == 3          # head_dim 96
    assert f(32, 32, 8, 128, 8192, 0) == 3      # Llama-shaped batch
    path = L.dec_decode_step_path               # which form: 0 short, 1 two launches, 2 three
    assert path(1, 4, 1, 64, 128, 0) == 0 and path(8, 64, 8, 128, 512, 0) == 0
    assert path(32, 32, 8, 128, 8192, 0) == 2   # no device to run the cooperative form here


def test_workspace_size_formula(L):
    for (B, Hq, Hkv, D, parts) in ((1, 4, 1, 64, 1), (32, 32, 8, 128, 152), (256, 16, 4, 128, 148)):
        G = Hq // Hkv
        slots = 5 * parts + B * Hkv
        pre = (256 + slots * G * D * 4 + slots * G * 4 + 15) // 16 * 16
        flags = (pre + (B + 1) * 4 + 15) // 16 * 16  # one completion word per piece
        raw = flags + 5 * parts * 4
        assert L.dec_attn_workspace_bytes(B, Hq, Hkv, D, 100, parts) == (raw + 255) // 256 * 256


def test_contract_sizing_helpers(L):
    """dec_pick_num_splits and dec_decode_workspace_bytes (host only, given the SM count)."""
    pick = L.dec_pick_num_splits
    assert pick(32, 8, 8192, 152) == 152          # Llama-shaped batch: one CTA per SM
    assert pick(1, 8, 131072, 152) == 152         # one long sequence
    assert pick(1, 1, 128, 152) == 2              # 128 rows: two blocks of 64
    assert pick(1, 1, 1, 152) == 1
    assert pick(0, 8, 100, 152) == 1 and pick(4, 8, 0, 152) == 1
    assert pick(256, 4, 14187, 148) == 148        # another SM count
    ws = L.dec_decode_workspace_bytes
    for (B, Hq, D, P) in ((32, 32, 128, 152), (256, 16, 128, 152), (1, 4, 64, 7), (3, 12, 64, 20)):
        got = ws(B, Hq, D, P)
        # at least the exact size of every supported grouping at every split count up to P
        for Hkv in range(1, Hq + 1):
            if Hq % Hkv or Hq // Hkv > 8:
                continue
            for parts in (1, P // 2 or 1, P):
                assert got >= L.dec_attn_workspace_bytes(B, Hq, Hkv, D, 100, parts), (B, Hq, Hkv, parts)
        # and equal to the largest of them (the group of 8, or of Hq when Hq < 8)
        assert got == max(L.dec_attn_workspace_bytes(B, Hq, h, D, 100, P)
                          for h in range(1, Hq + 1) if Hq % h == 0 and Hq // h <= 8)
    assert ws(-1, 8, 128, 4) == 0 and ws(2, 0, 128, 4) == 0 and ws(2, 8, 96, 4) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dsa.rmsnorm_residual(x, torch.ones(64, dtype=torch.bfloat16))


def test_norm_linear_rejects(L):
    X, R, NW = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    W, Y, H = ctypes.c_void_p(4 << 20), ctypes.c_void_p(5 << 20), ctypes.c_void_p(6 << 20)
    call = lambda *a: _st(L, "dec_norm_linear", *a)
    st, msg = call(X, R, NW, H, W, Y, 4, 100, 256, 1e-6, 0, None, None)
    assert st == 2 and "N" in msg
    st, msg = call(X, R, NW, H, W, Y, 4, 256, 96, 1e-6, 0, None, None)
    assert st == 2 and "K" in msg
    st, msg = call(X, R, NW, H, W, Y, 4, 256, 256, -1.0, 0, None, None)
    assert st == 1 and "eps" in msg
    st, msg = call(None, R, NW, H, W, Y, 4, 256, 256, 1e-6, 0, None, None)
    assert st == 1 and "non-null" in msg
    st, msg = call(X, R, None, H, W, Y, 4, 256, 256, 1e-6, 0, None, None)
    assert st == 1 and "non-null" in msg
    st, msg = call(X, R, NW, ctypes.c_void_p((6 << 20) + 8), W, Y, 4, 256, 256, 1e-6, 0, None,
                   None)
    assert st == 1 and "aligned" in msg
    st, msg = call(X, R, NW, ctypes.c_void_p((2 << 20) + 512), W, Y, 4, 256, 256, 1e-6, 0, None,
                   None)
    assert st == 1 and "h_out" in msg  # h_out inside the residual: other CTAs still read it
    st, msg = call(X, R, NW, H, W, ctypes.c_void_p((1 << 20) + 256), 4, 256, 256, 1e-6, 0, None,
                   None)
    assert st == 1 and "overlap" in msg  # y inside x
    st, msg = call(X, R, NW, H, W, Y, 4, 256, 256, 1e-6, 5, None, None)
    assert st == 1 and "k_split" in msg
    st, _ = call(None, None, None, None, None, None, 0, 256, 256, 1e-6, 0, None, None)
    assert st == 0  # B == 0 is a no-op


def test_norm_qkv_rejects(L):
    X, NW, WQ = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    Q, KC, VC, P = (ctypes.c_void_p(4 << 20), ctypes.c_void_p(5 << 20), ctypes.c_void_p(6 << 20),
                    ctypes.c_void_p(7 << 20))
    call = lambda *a: _st(L, "dec_norm_qkv_proj_rope_append", *a)
    st, msg = call(X, None, NW, None, WQ, None, None, Q, KC, VC, P, 2, 256, 8, 2, 64, 16, 1e4, 0,
                   None, 1e-6, None, None)
    assert st == 2 and "128" in msg  # head_dim 64 has no fused rotation
    st, msg = call(X, None, NW, None, WQ, None, None, ctypes.c_void_p((1 << 20) + 512), KC, VC, P,
                   2, 256, 8, 2, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 1 and "overlap" in msg  # q_out inside x
    st, msg = call(X, None, NW, ctypes.c_void_p((4 << 20) + 256), WQ, None, None, Q, KC, VC, P,
                   2, 256, 8, 2, 128, 16, 1e4, 0, None, 1e-6, None, None)
    assert st == 1 and "h_out" in msg


def test_linear_rejects(L):
    X, W, Y = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    st, msg = _st(L, "dec_linear", X, W, None, Y, 4, 100, 256, 0, None, None)
    assert st == 2 and "N" in msg  # N not a multiple of 128
    st, msg = _st(L, "dec_linear", X, W, None, Y, 4, 256, 96, 0, None, None)
    assert st == 2 and "K" in msg  # K not a multiple of 64
    st, _ = _st(L, "dec_linear", X, W, None, Y, -1, 256, 256, 0, None, None)
    assert st == 1
    st, _ = _st(L, "dec_linear", X, None, None, Y, 4, 256, 256, 0, None, None)
    assert st == 1
    st, msg = _st(L, "dec_linear", ctypes.c_void_p((1 << 20) + 8), W, None, Y, 4, 256, 256, 0,
                  None, 0, None)
    assert st == 1 and "aligned" in msg
    st, msg = _st(L, "dec_linear", X, W, None, ctypes.c_void_p((1 << 20) + 1024), 4, 256, 256,
                  0, None, None)
    assert st == 1 and "overlap" in msg  # y inside x
    st, msg = _st(L, "dec_linear", X, W, ctypes.c_void_p((3 << 20) + 64), Y, 4, 256, 256, 0,
                  None, 0, None)
    assert st == 1 and "residual" in msg  # residual partly overlapping y
    st, _ = _st(L, "dec_linear", None, None, None, None, 0, 256, 256, 0, None, None)
    assert st == 0  # B == 0 is a no-op
    for bad in (-1, 9, 5):  # 5 > K / 64 = 4
        st, msg = _st(L, "dec_linear", X, W, None, Y, 4, 256, 256, bad, None, None)
        assert st == 1 and "k_split" in msg
    nb, sp = ctypes.c_int(), ctypes.c_int()
    st, _ = _st(L, "dec_linear_plan", 0, 256, 256, ctypes.byref(nb), ctypes.byref(sp))
    assert st == 0 and nb.value == 16 and sp.value == 1
    for B, tile in ((1, 16), (16, 16), (17, 32), (33, 64), (65, 128), (129, 256), (1000, 256)):
        assert L.dec_linear_plan(B, 256, 256, ctypes.byref(nb), None) == 0 and nb.value == tile
    assert L.dec_linear_plan(4, 100, 256, None, None) == 2


def test_sublayer_rejects(L):
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(12)]
    x, res, nw, wqkv, wo, kc, vc, pos, lens, out, ws = p[:11]
    def call(B=2, hidden=1024, Hq=8, Hkv=2, D=128, window=0, eps=1e-6, ws_bytes=1 << 30,
             q_norm=None, k_norm=None, work=ws, o=out):
        return _st(L, "dec_attn_sublayer", x, res, nw, hidden, eps, wqkv, wo, q_norm, k_norm, kc,
                   vc, pos, lens, o, B, Hq, Hkv, D, 64, 64, 1e4, 0, None, 0.0, window, 4, work,
                   ws_bytes, None)
    st, msg = call(hidden=1000)
    assert st == 2 and "hidden" in msg
    st, msg = call(Hq=3, Hkv=1, D=64)
    assert st == 2 and "multiple of 128" in msg  # (3 + 2) * 64 = 320
    st, _ = call(window=-1)
    assert st == 1
    st, _ = call(eps=-1.0)
    assert st == 1
    st, msg = call(q_norm=p[11])
    assert st == 1 and "both" in msg
    st, msg = call(o=ctypes.c_void_p((1 << 24) + 256))
    assert st == 1 and "overlap" in msg
    st, _ = call(work=None)
    assert st == 3
    need = L.dec_attn_sublayer_workspace_bytes(2, 1024, 8, 2, 128, 64, 4)
    assert need >= L.dec_attn_workspace_bytes(2, 8, 2, 128, 64, 4) + 2 * 1024 * 2
    st, msg = call(ws_bytes=need - 256)
    assert st == 3 and "needed" in msg
    st, _ = call(B=0)
    assert st == 0


def test_sublayer_layout(L):
    off = (ctypes.c_size_t * 5)()
    B, hidden, Hq, Hkv, D = 32, 4096, 32, 8, 128
    assert L.dec_attn_sublayer_layout(B, hidden, Hq, Hkv, D, 8192, 152, off) == 0
    o = list(off)
    assert all(v % 256 == 0 for v in o)
    assert o[0] >= L.dec_attn_workspace_bytes(B, Hq, Hkv, D, 8192, 152)
    assert o[1] - o[0] >= B * hidden * 2
    assert o[2] - o[1] >= B * (Hq + 2 * Hkv) * D * 2
    assert o[3] - o[2] >= B * Hq * D * 2
    assert o[4] - o[3] >= B * Hq * D * 2
    assert o[4] == L.dec_attn_sublayer_workspace_bytes(B, hidden, Hq, Hkv, D, 8192, 152)


def test_sample_rejects(L):
    Z, T, U, I = (ctypes.c_void_p(k << 20) for k in (1, 2, 3, 4))
    def call(B=2, V=1000, pen=1.0, temp=1.0, p=0.9, k=0, ids=None, Lid=0, u=U, logits=Z):
        return _st(L, "dec_sample", logits, ids, Lid, u, T, B, V, pen, temp, p, k, None)
    assert call(B=-1)[0] == 1
    assert call(B=70000)[0] == 2
    assert call(V=0)[0] == 1
    assert call(V=10_000_000)[0] == 2
    assert call(V=262145)[0] == 2  # above 16 slices of 16384
    assert call(pen=0.0)[0] == 1
    assert call(temp=float("nan"))[0] == 1
    assert call(p=0.0)[0] == 1 and call(p=1.5)[0] == 1
    assert call(k=-1)[0] == 1
    assert call(Lid=4)[0] == 1  # ids missing
    assert call(u=None)[0] == 1  # sampling needs the uniforms
    st, msg = call(logits=ctypes.c_void_p((1 << 20) + 2))
    assert st == 1 and "aligned" in msg
    assert call(B=0, logits=None)[0] == 0


def test_rope_table_builder_matches_the_oracle(L):
    """dec_rope_inv_freq is host code: its tables against the oracle's, on the CPU."""
    import numpy as np
    from oracle import decode_ref as O
    for D in (64, 128):
        for theta in (1e4, 5e5, 1e6):
            for scaling in ("none", "linear", "ntk"):
                for factor in (1.0, 2.0, 4.0, 8.0, 32.0):
                    got = dsa.rope_inv_freq(D, theta, scaling, factor).numpy()
                    ref = O.rope_scaled_inv_freq(D, np.float32(theta), scaling, factor)
                    assert got.shape == (D // 2,)
                    rel = np.max(np.abs(got - ref) / ref)
                    assert rel <= 1e-14, (D, theta, scaling, factor, rel)
                    assert np.all(got <= 1.0) and np.all(got > 0.0)


def test_rope_table_builder_rejects(L):
    buf = (ctypes.c_double * 64)()
    assert _st(L, "dec_rope_inv_freq", 96, 1e4, 0, 1.0, buf)[0] == 2      # head_dim
    assert _st(L, "dec_rope_inv_freq", 128, 0.0, 0, 1.0, buf)[0] == 1     # theta
    assert _st(L, "dec_rope_inv_freq", 128, 1e4, 1, 0.5, buf)[0] == 1     # factor < 1
    assert _st(L, "dec_rope_inv_freq", 128, 1e4, 2, float("inf"), buf)[0] == 1
    assert _st(L, "dec_rope_inv_freq", 128, 1e4, 9, 2.0, buf)[0] == 1     # unknown scaling
    assert _st(L, "dec_rope_inv_freq", 128, 1e4, 1, 2.0, None)[0] == 1    # no output
    assert _st(L, "dec_rope_inv_freq", 128, 1e4, 0, 0.0, buf)[0] == 0     # factor unread
    with pytest.raises(ValueError):
        dsa.rope_inv_freq(128, 1e4, "dynamic", 2.0)
    with pytest.raises(ValueError):
        dsa._freq([0.5] * 63, 128)


def test_yarn_table_builder_matches_the_oracle(L):
    """dec_rope_yarn_inv_freq (host code) against the oracle's YaRN table and factor."""
    import math
    import numpy as np
    from oracle import decode_ref as O
    for D in (64, 128):
        for theta in (1e4, 5e5):
            for s in (1.0, 2.0, 8.0, 32.0):
                for ctx, a, b in ((4096, 1.0, 32.0), (8192, 1.0, 32.0), (2048, 0.5, 16.0)):
                    got = dsa.rope_inv_freq(D, theta, "yarn", s, ctx, a, b).numpy()
                    ref = O.rope_scaled_inv_freq(D, np.float32(theta), "yarn", s, ctx, a, b)
                    rel = np.max(np.abs(got - ref) / ref)
                    assert rel <= 1e-14, (D, theta, s, ctx, rel)
            m = O.yarn_attention_factor(s)
            assert abs(dsa.yarn_softmax_scale(D, s) - m * m / math.sqrt(D)) <= 1e-6 * m * m
    buf = (ctypes.c_double * 64)()
    assert _st(L, "dec_rope_yarn_inv_freq", 96, 1e4, 2.0, 4096, 1.0, 32.0, buf, None)[0] == 2
    assert _st(L, "dec_rope_yarn_inv_freq", 128, 1e4, 0.5, 4096, 1.0, 32.0, buf, None)[0] == 1
    assert _st(L, "dec_rope_yarn_inv_freq", 128, 1e4, 2.0, 0, 1.0, 32.0, buf, None)[0] == 1
    assert _st(L, "dec_rope_yarn_inv_freq", 128, 1e4, 2.0, 4096, 32.0, 1.0, buf, None)[0] == 1
    assert _st(L, "dec_rope_yarn_inv_freq", 128, -1.0, 2.0, 4096, 1.0, 32.0, buf, None)[0] == 1
    sc = ctypes.c_float()
    assert _st(L, "dec_rope_yarn_softmax_scale", 96, 2.0, ctypes.byref(sc))[0] == 2
    assert _st(L, "dec_rope_yarn_softmax_scale", 128, 0.9, ctypes.byref(sc))[0] == 1
    assert _st(L, "dec_rope_yarn_softmax_scale", 128, 2.0, None)[0] == 1
    mult = ctypes.c_float()
    assert _st(L, "dec_rope_yarn_inv_freq", 64, 1e4, 8.0, 4096, 1.0, 32.0, buf,
               ctypes.byref(mult))[0] == 0
    assert abs(dsa.yarn_softmax_scale(64, 8.0) - mult.value / 8.0) <= 1e-6 * mult.value
