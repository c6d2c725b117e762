"""GB300-native (sm_103a) decode-step attention block.

A thin ctypes binding over ``libdecattn.so``, whose C ABI is declared in
``include/decattn.h``. This module only checks tensor metadata, passes raw device
pointers, sizes and torch's current CUDA stream, and turns status codes into
exceptions: every step of the block runs in the library's CUDA kernels. There is
no CPU path; without the built library every call raises.

Steps (fusedtok 1.0.1 README, "Operators" and "Usage"; cutileGPT README, "Why
tiles" and "The current runtime includes"):

* :func:`rmsnorm_residual`      RMSNorm with a fused residual add;
* :func:`qknorm_rope_kv_append` per-head QK-RMSNorm, RoPE (NeoX / interleaved) at
  each sequence's position, K/V append into a contiguous cache; the frequency table
  may be a context-extension one (:func:`rope_inv_freq`: linear interpolation or the
  NTK-aware base; PyGPUkit 0.2.18 page, "Positional Encoding Operations");
* :func:`gqa_decode_attn`       single-query GQA attention with the split-KV pass
  (:func:`gqa_decode_split`) and the log-sum-exp merge (:func:`split_merge`);
* :func:`decode_step`           the whole block on one stream: K1 + K2 (one launch),
  the split pass and the merge, or for short contexts a single launch.

Around the block (cutileGPT README, "The current runtime includes": packed QKV
projections, fused down-projection + residual epilogues):

* :func:`linear`                y = x W^T (+ residual) on the tensor cores;
* :func:`norm_linear`, :func:`norm_qkv_proj_rope_append`  projections with the
  RMSNorm as their prologue;
* :func:`attn_sublayer`         RMSNorm -> packed QKV projection -> rotation and
  append -> attention -> output projection + residual, on one stream.

The sampling side of the decode step (fusedtok README, "Operators": repetition
penalty, temperature, top-k / top-p sampling, decode_step):

* :func:`sample`                penalty -> temperature -> top-k -> top-p -> draw,
  one launch for a batch of rows.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdecattn.so")

NEOX = 0
INTERLEAVED = 1
_LAYOUTS = {"neox": NEOX, "interleaved": INTERLEAVED, NEOX: NEOX, INTERLEAVED: INTERLEAVED}

DEVERR_LEN_CLAMPED = 0x1
DEVERR_POS_SKIPPED = 0x2
DEVERR_WAIT_TIMEOUT = 0x4

WORKSPACE_HEADER_BYTES = 256

# C ABI: name -> (restype, argtypes)
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
EXPORTS = {
    "dec_rmsnorm_residual": (_I, [_P, _P, _P, _P, _I, _I, _F, _P]),
    "dec_rope_inv_freq": (_I, [_I, _F, _I, _F, ctypes.POINTER(ctypes.c_double)]),
    "dec_rope_yarn_inv_freq": (_I, [_I, _F, _F, _I, _F, _F, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(_F)]),
    "dec_rope_yarn_softmax_scale": (_I, [_I, _F, ctypes.POINTER(_F)]),
    "dec_qknorm_rope_kv_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F,
                                       _I, _P, _F, _P, _P]),
    "dec_qknorm_rope_kv_append_out": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                           _I, _F, _I, _P, _F, _P, _P]),
    "dec_decode_step_launches": (_I, [_I, _I, _I, _I, _I, _I]),
    "dec_decode_step_path": (_I, [_I, _I, _I, _I, _I, _I]),
    "dec_attn_default_parts": (_I, [_I, _I, _I, _I]),
    "dec_attn_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I]),
    "dec_pick_num_splits": (_I, [_I, _I, _I, _I]),
    "dec_decode_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "dec_gqa_decode_split": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "dec_split_merge": (_I, [_P, _Z, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "dec_gqa_decode_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "dec_gqa_decode_attn_window": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                        _P, _Z, _P]),
    "dec_decode_step": (_I, [_P, _P, _P, _P, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                             _I, _I, _I, _I, _I, _I, _F, _I, _P, _F, _I, _I, _P, _Z, _P]),
    "dec_gqa_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P]),
    "dec_linear_plan": (_I, [_I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "dec_linear": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "dec_qkv_proj_rope_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                      _F, _I, _P, _F, _P, _P]),
    "dec_norm_linear": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _I, _P, _P]),
    "dec_norm_qkv_proj_rope_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                                           _I, _I, _I, _I, _F, _I, _P, _F, _P, _P]),
    "dec_attn_sublayer_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "dec_attn_sublayer_layout": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_Z)]),
    "dec_attn_sublayer": (_I, [_P, _P, _P, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               _I, _I, _I, _I, _I, _I, _F, _I, _P, _F, _I, _I, _P, _Z, _P]),
    "dec_sample": (_I, [_P, _P, _I, _P, _P, _I, _I, _F, _F, _F, _I, _P]),
    "dec_diag_wait_timeout": (_I, [_P, _P]),
    "dec_status_string": (ctypes.c_char_p, [_I]),
    "dec_last_error": (ctypes.c_char_p, []),
    "dec_version": (_I, []),
}

_lib = None


class DecAttnError(RuntimeError):
    """A non-zero status from the C ABI."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libdecattn.so (once). Raises if the CUDA library was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m decode_step_attention_gb300.build` "
                "(there is no CPU fallback)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _call(name: str, *args) -> None:
    L = lib()
    st = getattr(L, name)(*args)
    if st != 0:
        raise DecAttnError(name, st, f"{L.dec_status_string(st).decode()}: {L.dec_last_error().decode()}")


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name: str, dtype, shape=None, host: bool = False) -> None:
    """Checks a tensor argument. ``host``: the kernels may also reach it in pinned
    (page-locked, mapped) host memory, which they then read or write across the host
    link themselves; the library confirms the mapping before it launches."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda and not (host and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" +
                         (" or a pinned host tensor" if host else "") + " (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


BF16 = torch.bfloat16
I32 = torch.int32


def _empty(shape, dtype, like):
    """A new tensor where ``like`` lives: on its device, or pinned on the host."""
    if like.is_cuda:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return torch.empty(shape, dtype=dtype, pin_memory=True)


ROPE_SCALINGS = {"none": 0, "linear": 1, "ntk": 2}


def _freq(inv_freq, D: int):
    """A RoPE frequency table as the C calls take it: None, or D/2 doubles in host
    memory (kept alive by the caller's reference for the length of the call)."""
    if inv_freq is None:
        return None
    if isinstance(inv_freq, torch.Tensor):
        if inv_freq.is_cuda:
            raise ValueError("inv_freq must be on the host (the library reads it during the call)")
        inv_freq = inv_freq.double().tolist()
    vals = [float(v) for v in inv_freq]
    if len(vals) != D // 2:
        raise ValueError(f"inv_freq must hold D/2 = {D // 2} values, got {len(vals)}")
    return (ctypes.c_double * len(vals))(*vals)


def rope_inv_freq(D: int, theta: float, scaling: str = "none", factor: float = 1.0,
                  original_context: int = 4096, alpha: float = 1.0, beta: float = 32.0):
    """The RoPE frequency table [D/2] (float64, host) for context extension: "linear"
    position interpolation, the "ntk"-aware base or "yarn" (with ``original_context``,
    ``alpha`` and ``beta``), by ``factor``; "none" gives theta^(-2i/D). Pass it as
    ``inv_freq`` to any call that rotates; with "yarn" also pass
    ``scale=yarn_softmax_scale(D, factor)`` to the calls that attend."""
    arr = (ctypes.c_double * (int(D) // 2))()
    if scaling == "yarn":
        _call("dec_rope_yarn_inv_freq", int(D), float(theta), float(factor),
              int(original_context), float(alpha), float(beta), arr, None)
    elif scaling in ROPE_SCALINGS:
        _call("dec_rope_inv_freq", int(D), float(theta), ROPE_SCALINGS[scaling], float(factor),
              arr)
    else:
        raise ValueError(f"scaling must be one of {sorted(ROPE_SCALINGS) + ['yarn']}")
    return torch.tensor(list(arr), dtype=torch.float64)


def yarn_softmax_scale(D: int, factor: float) -> float:
    """The softmax scale that carries YaRN's attention temperature: m^2 / sqrt(D), m =
    0.1 ln(factor) + 1 (dec_rope_yarn_softmax_scale)."""
    scale = ctypes.c_float()
    _call("dec_rope_yarn_softmax_scale", int(D), float(factor), ctypes.byref(scale))
    return float(scale.value)


# ------------------------------------------------------------------- K1 ---
def rmsnorm_residual(x, weight, residual=None, eps: float = 1e-6, out=None, stream=None):
    """y = RMSNorm(x + residual) * weight; residual <- x + residual (in place) when given."""
    _need(x, "x", BF16, host=True)
    B, hidden = x.shape
    _need(weight, "weight", BF16, (hidden,), host=True)
    if residual is not None:
        _need(residual, "residual", BF16, (B, hidden), host=True)
    if out is None:
        out = _empty((B, hidden), BF16, x)
    _need(out, "out", BF16, (B, hidden), host=True)
    _call("dec_rmsnorm_residual", _ptr(x), _ptr(residual), _ptr(weight), _ptr(out), B, hidden,
          float(eps), _stream(stream))
    return out


# ------------------------------------------------------------------- K2 ---
def qknorm_rope_kv_append(q, k_new, v_new, k_cache, v_cache, pos, theta: float, layout="neox",
                          q_norm_w=None, k_norm_w=None, eps: float = 1e-6, error_word=None,
                          stream=None, q_out=None, inv_freq=None):
    """QK-norm (optional) + RoPE at pos[b]; q rotated in place (or into ``q_out``,
    leaving q as is), K/V written to slot pos[b]. ``inv_freq``: a frequency table
    (:func:`rope_inv_freq`, or any D/2 values in [0, 1]) in place of theta^(-2i/D).
    Returns the rotated q."""
    _need(q, "q", BF16, host=True)
    B, Hq, D = q.shape
    _need(k_cache, "k_cache", BF16)
    _, Hkv, T_cap, _ = k_cache.shape
    _need(v_cache, "v_cache", BF16, (B, Hkv, T_cap, D))
    _need(k_cache, "k_cache", BF16, (B, Hkv, T_cap, D))
    _need(k_new, "k_new", BF16, (B, Hkv, D), host=True)
    _need(v_new, "v_new", BF16, (B, Hkv, D), host=True)
    _need(pos, "pos", I32, (B,), host=True)
    for n, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _need(w, n, BF16, (D,), host=True)
    if error_word is not None:
        _need(error_word, "error_word", I32, host=True)
    args = (_ptr(k_new), _ptr(v_new), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(k_cache),
            _ptr(v_cache), _ptr(pos), B, Hq, Hkv, D, T_cap, float(theta), _LAYOUTS[layout],
            _freq(inv_freq, D), float(eps), _ptr(error_word), _stream(stream))
    if q_out is None:
        _call("dec_qknorm_rope_kv_append", _ptr(q), *args)
        return q
    _need(q_out, "q_out", BF16, (B, Hq, D), host=True)
    _call("dec_qknorm_rope_kv_append_out", _ptr(q), _ptr(q_out), *args)
    return q_out


# -------------------------------------------------------------- K3 + K4 ---
def default_parts(B: int, Hkv: int, D: int, max_len: int) -> int:
    return int(lib().dec_attn_default_parts(B, Hkv, D, max_len))


def attn_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, max_len: int, num_parts: int = 0) -> int:
    return int(lib().dec_attn_workspace_bytes(B, Hq, Hkv, D, max_len, num_parts))


def alloc_workspace(B: int, Hq: int, Hkv: int, D: int, max_len: int, num_parts: int = 0,
                    device=None) -> torch.Tensor:
    """A zeroed uint8 workspace of the size the attention call needs."""
    n = attn_workspace_bytes(B, Hq, Hkv, D, max_len, num_parts)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def device_errors(workspace: torch.Tensor) -> int:
    """The device error word at the head of a workspace (reads it back: synchronises)."""
    return int(workspace[:4].view(torch.int32).item())


def _attn_dims(q, k_cache, v_cache, lens, q_host=False):
    _need(q, "q", BF16, host=q_host)
    B, Hq, D = q.shape
    _need(k_cache, "k_cache", BF16)
    if k_cache.dim() != 4 or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError(f"k_cache shape {tuple(k_cache.shape)} does not match q {tuple(q.shape)}")
    Hkv, T_cap = k_cache.shape[1], k_cache.shape[2]
    _need(v_cache, "v_cache", BF16, (B, Hkv, T_cap, D))
    _need(lens, "lens", I32, (B,), host=True)
    return B, Hq, Hkv, D, T_cap


def gqa_decode_split(q, k_cache, v_cache, lens, workspace, max_len=None, scale: float = 0.0,
                     num_parts: int = 0, stream=None):
    """The split pass alone: partials into ``workspace``."""
    B, Hq, Hkv, D, T_cap = _attn_dims(q, k_cache, v_cache, lens)
    max_len = T_cap if max_len is None else int(max_len)
    _need(workspace, "workspace", torch.uint8)
    _call("dec_gqa_decode_split", _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), B, Hq, Hkv,
          D, T_cap, max_len, float(scale), int(num_parts), _ptr(workspace), workspace.numel(),
          _stream(stream))


def split_merge(workspace, lens, out, Hkv: int, T_cap: int, max_len=None, num_parts: int = 0,
                stream=None):
    """The merge pass alone: partials in ``workspace`` -> bf16 ``out`` [B, Hq, D]."""
    _need(out, "out", BF16, host=True)
    B, Hq, D = out.shape
    _need(lens, "lens", I32, (B,), host=True)
    _need(workspace, "workspace", torch.uint8)
    max_len = T_cap if max_len is None else int(max_len)
    _call("dec_split_merge", _ptr(workspace), workspace.numel(), _ptr(lens), _ptr(out), B, Hq,
          Hkv, D, T_cap, max_len, int(num_parts), _stream(stream))
    return out


def gqa_decode_attn(q, k_cache, v_cache, lens, max_len=None, workspace=None, out=None,
                    scale: float = 0.0, num_parts: int = 0, stream=None, window: int = 0):
    """Single-query GQA decode attention: split pass + merge, or for short contexts with
    ``num_parts`` = 0 (where :func:`decode_step_launches` reports 1) both in one launch.
    Returns ``out`` [B, Hq, D].

    ``window`` > 0 restricts sequence b to its last min(lens[b], window) tokens."""
    B, Hq, Hkv, D, T_cap = _attn_dims(q, k_cache, v_cache, lens)
    max_len = T_cap if max_len is None else int(max_len)
    if workspace is None:
        workspace = alloc_workspace(B, Hq, Hkv, D, max_len, num_parts, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", BF16, (B, Hq, D), host=True)
    if window:
        _call("dec_gqa_decode_attn_window", _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens),
              _ptr(out), B, Hq, Hkv, D, T_cap, max_len, int(window), float(scale), int(num_parts),
              _ptr(workspace), workspace.numel(), _stream(stream))
    else:
        _call("dec_gqa_decode_attn", _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), _ptr(out),
              B, Hq, Hkv, D, T_cap, max_len, float(scale), int(num_parts), _ptr(workspace),
              workspace.numel(), _stream(stream))
    return out


# -------------------------------------------------------- the whole block ---
STEP_SHORT, STEP_STREAM, STEP_THREE = 0, 1, 2


def decode_step_path(B: int, Hq: int, Hkv: int, D: int, max_len: int, window: int = 0) -> int:
    """Which form :func:`decode_step` takes for this shape on the current device:
    STEP_SHORT (one launch, the short-context kernel), STEP_STREAM (two launches: K1 + K2,
    then the split pass and its merge in one cooperative launch) or STEP_THREE (three
    launches: K1 + K2, split pass, merge)."""
    return int(lib().dec_decode_step_path(B, Hq, Hkv, D, max_len, window))


def decode_step_launches(B: int, Hq: int, Hkv: int, D: int, max_len: int, window: int = 0) -> int:
    """Kernel launches :func:`decode_step` makes for this shape: 1, 2 or 3 (see
    :func:`decode_step_path`)."""
    return int(lib().dec_decode_step_launches(B, Hq, Hkv, D, max_len, window))



def decode_step(x, residual, norm_w, y, q, k_new, v_new, k_cache, v_cache, pos, lens, out,
                workspace, theta: float, layout="neox", q_norm_w=None, k_norm_w=None,
                eps: float = 1e-6, max_len=None, scale: float = 0.0, num_parts: int = 0,
                stream=None, window: int = 0, inv_freq=None):
    """K1 + K2 (one launch) -> K3 -> K4 on one stream, or for short contexts the whole
    step in one launch (:func:`decode_step_launches`); ``window`` > 0 gives
    sliding-window attention, ``inv_freq`` a RoPE frequency table."""
    B, Hq, Hkv, D, T_cap = _attn_dims(q, k_cache, v_cache, lens, q_host=True)
    _need(x, "x", BF16, host=True)
    hidden = x.shape[1]
    _need(y, "y", BF16, (B, hidden), host=True)
    _need(norm_w, "norm_w", BF16, (hidden,), host=True)
    if residual is not None:
        _need(residual, "residual", BF16, (B, hidden), host=True)
    _need(k_new, "k_new", BF16, (B, Hkv, D), host=True)
    _need(v_new, "v_new", BF16, (B, Hkv, D), host=True)
    _need(pos, "pos", I32, (B,), host=True)
    _need(out, "out", BF16, (B, Hq, D), host=True)
    _need(workspace, "workspace", torch.uint8)
    for n, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _need(w, n, BF16, (D,), host=True)
    max_len = T_cap if max_len is None else int(max_len)
    _call("dec_decode_step", _ptr(x), _ptr(residual), _ptr(norm_w), _ptr(y), hidden, float(eps),
          _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(k_cache),
          _ptr(v_cache), _ptr(pos), _ptr(lens), _ptr(out), B, Hq, Hkv, D, T_cap, max_len,
          float(theta), _LAYOUTS[layout], _freq(inv_freq, D), float(scale), int(window),
          int(num_parts), _ptr(workspace), workspace.numel(), _stream(stream))
    return out


# ------------------------------------------------------------ projections ---
def linear_plan(B: int, N: int, K: int):
    """(batch tile, K split) :func:`linear` uses for this shape on this device; the K
    split is the number of CTAs (one cluster) that share each output tile."""
    nb, sp = _I(), _I()
    _call("dec_linear_plan", B, N, K, ctypes.byref(nb), ctypes.byref(sp))
    return nb.value, sp.value


def linear(x, w, residual=None, out=None, error_word=None, stream=None, k_split: int = 0):
    """y = x w^T (+ residual): x [B, K], w [N, K], residual / out [B, N], all bf16.
    ``error_word`` (optional) is a device tensor whose first 4 bytes collect DEVERR_*
    bits; ``k_split`` 0 chooses the K split, 1 .. 8 forces it."""
    _need(x, "x", BF16)
    _need(w, "w", BF16)
    B, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError(f"w has shape {tuple(w.shape)}, expected (N, {K})")
    if residual is not None:
        _need(residual, "residual", BF16, (B, N), host=True)
    if out is None:
        out = torch.empty((B, N), dtype=BF16, device=x.device)
    _need(out, "out", BF16, (B, N), host=True)
    if error_word is not None and not (error_word.is_cuda or error_word.is_pinned()):
        raise ValueError("error_word must be a CUDA tensor or a pinned host tensor")
    _call("dec_linear", _ptr(x), _ptr(w), _ptr(residual), _ptr(out), B, N, K, int(k_split),
          _ptr(error_word), _stream(stream))
    return out


def _norm_inputs(x, residual, norm_w, h_out):
    _need(x, "x", BF16)
    B, K = x.shape
    if residual is not None:
        _need(residual, "residual", BF16, (B, K))
    _need(norm_w, "norm_w", BF16, (K,))
    if h_out is not None:
        _need(h_out, "h_out", BF16, (B, K), host=True)
    return B, K


def norm_linear(x, w, norm_w, residual=None, h_out=None, eps: float = 1e-6, out=None,
                error_word=None, stream=None, k_split: int = 0):
    """y = RMSNorm(x + residual) w^T with the normalisation formed inside the projection
    (x, residual [B, K], norm_w [K], w [N, K], all bf16); ``h_out`` (optional) receives
    x + residual."""
    B, K = _norm_inputs(x, residual, norm_w, h_out)
    _need(w, "w", BF16)
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError(f"w has shape {tuple(w.shape)}, expected (N, {K})")
    if out is None:
        out = torch.empty((B, N), dtype=BF16, device=x.device)
    _need(out, "out", BF16, (B, N), host=True)
    _call("dec_norm_linear", _ptr(x), _ptr(residual), _ptr(norm_w), _ptr(h_out), _ptr(w),
          _ptr(out), B, N, K, float(eps), int(k_split), _ptr(error_word), _stream(stream))
    return out


def norm_qkv_proj_rope_append(x, w_qkv, norm_w, k_cache, v_cache, pos, theta: float,
                              layout="neox", residual=None, h_out=None, q_norm_w=None,
                              k_norm_w=None, eps: float = 1e-6, q_out=None, error_word=None,
                              stream=None, inv_freq=None):
    """The packed QKV projection of RMSNorm(x + residual) (formed in its prologue) with
    QK-norm + RoPE + K/V append as its epilogue (head_dim 128). Returns the rotated q."""
    B, hidden = _norm_inputs(x, residual, norm_w, h_out)
    _need(k_cache, "k_cache", BF16)
    Hkv, T_cap, D = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    _need(v_cache, "v_cache", BF16, (B, Hkv, T_cap, D))
    _need(w_qkv, "w_qkv", BF16)
    Hq = w_qkv.shape[0] // D - 2 * Hkv
    _need(w_qkv, "w_qkv", BF16, ((Hq + 2 * Hkv) * D, hidden))
    _need(pos, "pos", I32, (B,), host=True)
    if q_out is None:
        q_out = torch.empty(B, Hq, D, dtype=BF16, device=x.device)
    _need(q_out, "q_out", BF16, (B, Hq, D), host=True)
    for n, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _need(w, n, BF16, (D,), host=True)
    _call("dec_norm_qkv_proj_rope_append", _ptr(x), _ptr(residual), _ptr(norm_w), _ptr(h_out),
          _ptr(w_qkv), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(q_out), _ptr(k_cache),
          _ptr(v_cache), _ptr(pos), B, hidden, Hq, Hkv, D, T_cap, float(theta),
          _LAYOUTS[layout], _freq(inv_freq, D), float(eps), _ptr(error_word), _stream(stream))
    return q_out


def sublayer_workspace_bytes(B: int, hidden: int, Hq: int, Hkv: int, D: int, max_len: int,
                             num_parts: int = 0) -> int:
    return int(lib().dec_attn_sublayer_workspace_bytes(B, hidden, Hq, Hkv, D, max_len, num_parts))


def qkv_proj_rope_append(y, w_qkv, k_cache, v_cache, pos, theta: float, layout="neox",
                         q_norm_w=None, k_norm_w=None, eps: float = 1e-6, q_out=None,
                         error_word=None, stream=None, inv_freq=None):
    """The packed QKV projection of ``y`` [B, hidden] with QK-norm + RoPE + K/V append
    as its epilogue (head_dim 128). Returns the rotated q [B, Hq, 128]."""
    _need(y, "y", BF16)
    B, hidden = y.shape
    _need(k_cache, "k_cache", BF16)
    Hkv, T_cap, D = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    _need(v_cache, "v_cache", BF16, (B, Hkv, T_cap, D))
    _need(w_qkv, "w_qkv", BF16)
    Hq = w_qkv.shape[0] // D - 2 * Hkv
    _need(w_qkv, "w_qkv", BF16, ((Hq + 2 * Hkv) * D, hidden))
    _need(pos, "pos", I32, (B,))
    if q_out is None:
        q_out = torch.empty(B, Hq, D, dtype=BF16, device=y.device)
    _need(q_out, "q_out", BF16, (B, Hq, D))
    for n, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _need(w, n, BF16, (D,))
    _call("dec_qkv_proj_rope_append", _ptr(y), _ptr(w_qkv), _ptr(q_norm_w), _ptr(k_norm_w),
          _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(pos), B, hidden, Hq, Hkv, D, T_cap,
          float(theta), _LAYOUTS[layout], _freq(inv_freq, D), float(eps), _ptr(error_word),
          _stream(stream))
    return q_out


def sublayer_views(workspace, B: int, hidden: int, Hq: int, Hkv: int, D: int, max_len: int,
                   num_parts: int = 0) -> dict:
    """Views of the intermediates an :func:`attn_sublayer` call left in ``workspace``:
    y [B, hidden], qkv [B, (Hq + 2 Hkv) D] (head_dim 64 only), q_rot [B, Hq, D],
    attn [B, Hq, D]."""
    off = (_Z * 5)()
    _call("dec_attn_sublayer_layout", B, hidden, Hq, Hkv, D, max_len, num_parts, off)
    if workspace.numel() < off[4]:
        raise ValueError("workspace smaller than the sublayer layout")
    nqkv = (Hq + 2 * Hkv) * D

    def view(o, shape):
        n = 1
        for v in shape:
            n *= v
        return workspace[o:o + 2 * n].view(BF16).view(shape)

    return {"y": view(off[0], (B, hidden)), "qkv": view(off[1], (B, nqkv)),
            "q_rot": view(off[2], (B, Hq, D)), "attn": view(off[3], (B, Hq, D))}


def attn_sublayer(x, residual, norm_w, w_qkv, w_o, k_cache, v_cache, pos, lens, out, workspace,
                  theta: float, layout="neox", q_norm_w=None, k_norm_w=None, eps: float = 1e-6,
                  max_len=None, scale: float = 0.0, num_parts: int = 0, stream=None,
                  window: int = 0, inv_freq=None):
    """h = x + residual (kept in ``residual``); out = h + Attn(RMSNorm(h)) W_o^T with
    the packed QKV projection, rotation and append, and attention in between."""
    _need(x, "x", BF16, host=True)
    B, hidden = x.shape
    _need(k_cache, "k_cache", BF16)
    if k_cache.dim() != 4 or k_cache.shape[0] != B:
        raise ValueError(f"k_cache shape {tuple(k_cache.shape)} does not match B = {B}")
    Hkv, T_cap, D = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    _need(v_cache, "v_cache", BF16, (B, Hkv, T_cap, D))
    _need(w_qkv, "w_qkv", BF16)
    nqkv = w_qkv.shape[0]
    Hq = nqkv // D - 2 * Hkv
    _need(w_qkv, "w_qkv", BF16, ((Hq + 2 * Hkv) * D, hidden))
    _need(w_o, "w_o", BF16, (hidden, Hq * D))
    _need(norm_w, "norm_w", BF16, (hidden,), host=True)
    if residual is not None:
        _need(residual, "residual", BF16, (B, hidden), host=True)
    _need(pos, "pos", I32, (B,), host=True)
    _need(lens, "lens", I32, (B,), host=True)
    _need(out, "out", BF16, (B, hidden), host=True)
    _need(workspace, "workspace", torch.uint8)
    for n, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _need(w, n, BF16, (D,))
    max_len = T_cap if max_len is None else int(max_len)
    _call("dec_attn_sublayer", _ptr(x), _ptr(residual), _ptr(norm_w), hidden, float(eps),
          _ptr(w_qkv), _ptr(w_o), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(k_cache), _ptr(v_cache),
          _ptr(pos), _ptr(lens), _ptr(out), B, Hq, Hkv, D, T_cap, max_len, float(theta),
          _LAYOUTS[layout], _freq(inv_freq, D), float(scale), int(window), int(num_parts),
          _ptr(workspace), workspace.numel(), _stream(stream))
    return out


# ------------------------------------------------------------------ sampler ---
def sample(logits, sampled_ids=None, penalty: float = 1.0, temperature: float = 1.0,
           top_p: float = 1.0, top_k: int = 0, u=None, seed=None, out=None, stream=None):
    """One token per row of ``logits`` [B, V] (fp32): CTRL repetition penalty over the
    ids in ``sampled_ids`` [B, L] (int32, negative = padding), then greedy argmax when
    ``temperature`` <= 0, else softmax(z / temperature) -> top-k -> top-p -> a draw
    with the uniforms ``u`` [B] (fp32 in [0, 1)); when ``u`` is None they come from a
    CPU ``torch.Generator`` seeded with ``seed`` (0 if None). Returns int32 [B]."""
    _need(logits, "logits", torch.float32, host=True)
    B, V = logits.shape
    L = 0
    if sampled_ids is not None:
        _need(sampled_ids, "sampled_ids", I32, host=True)
        if sampled_ids.dim() != 2 or sampled_ids.shape[0] != B:
            raise ValueError(f"sampled_ids must be [B, L], got {tuple(sampled_ids.shape)}")
        L = sampled_ids.shape[1]
    if temperature > 0 and u is None:
        g = torch.Generator().manual_seed(0 if seed is None else int(seed))
        u = torch.rand(B, generator=g, dtype=torch.float32)
        u = u.to(logits.device) if logits.is_cuda else u.pin_memory()
    if u is not None:
        _need(u, "u", torch.float32, (B,), host=True)
    if out is None:
        out = _empty((B,), I32, logits)
    _need(out, "out", I32, (B,), host=True)
    _call("dec_sample", _ptr(logits), _ptr(sampled_ids) if L else None, L, _ptr(u), _ptr(out),
          B, V, float(penalty), float(temperature), float(top_p), int(top_k), _stream(stream))
    return out


# ------------------------------------------------------------ CUDA graph ---
class GraphBranch:
    """A step with its own copies in and out, captured by :class:`StepGraph` on a
    stream of its own. It depends on the main ``copies_in`` and ``prologue`` only and
    is joined back before the graph ends, so work that does not need the main step
    (the RMSNorm half of a decode step against its attention half, say) overlaps it.
    It is captured after the main step: the graph then launches the main step's
    kernels first, and a long main kernel that fills every SM (the split pass) is
    resident before the branch's small blocks take their place beside it. Captured the
    other way round, those blocks could reach the SMs first and hold the big one
    back. ``priority`` is the CUDA stream priority of the branch's stream (lower is
    more urgent)."""

    def __init__(self, step, copies_in=(), copies_out=(), priority: int = 0, **step_kwargs):
        self.step = step
        self.kwargs = step_kwargs
        self.copies_in = list(copies_in)
        self.copies_out = list(copies_out)
        self.priority = int(priority)


class StepGraph:
    """One :func:`decode_step` (or ``step``, e.g. :func:`attn_sublayer`) on fixed
    buffers, captured into a CUDA graph.

    ``replay()`` re-runs the kernels with a single graph launch, so the host cost of
    the step no longer adds to its latency. The first call on a device sets up
    per-device state, so the constructor runs the step once eagerly on a side stream
    before capturing it. Buffers are bound at capture: refill them in place
    (``copy_``) between replays. The kernels chain with programmatic dependent
    launch, which the graph keeps.

    ``copies_in`` / ``copies_out`` (optional) are lists of ``(src, dst)`` tensor
    pairs copied before / after the step inside the same graph — typically pinned
    host buffers to device buffers the step reads, and device results back to pinned
    host buffers — so one replay is a whole host-to-host decode step (read the host
    results after synchronising). Packing the step's inputs (and outputs) as views of
    one buffer makes that one copy each way. ``branches`` (optional) are
    :class:`GraphBranch` es captured on streams of their own beside the main step;
    ``prologue`` (optional, no arguments) runs on the main stream before they fork.
    """

    def __init__(self, copies_in=(), copies_out=(), step=None, branches=(), prologue=None,
                 **step_kwargs):
        self.step = decode_step if step is None else step
        self.prologue = prologue
        self.kwargs = step_kwargs
        self.copies_in = list(copies_in)
        self.copies_out = list(copies_out)
        self.branches = list(branches)
        pairs = self.copies_in + self.copies_out
        for br in self.branches:
            pairs += br.copies_in + br.copies_out
        for src, dst in pairs:
            if src.shape != dst.shape or src.dtype != dst.dtype:
                raise ValueError("copy pairs need the same shape and dtype")
            for t in (src, dst):
                if not t.is_cuda and not t.is_pinned():
                    raise ValueError("host buffers in copy pairs must be pinned")
        self._streams = [torch.cuda.Stream(priority=br.priority) for br in self.branches]
        cur = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            self._body()
        cur.wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()

    @staticmethod
    def _copies(pairs):
        for src, dst in pairs:
            dst.copy_(src, non_blocking=True)

    def _body(self):
        main = torch.cuda.current_stream()
        self._copies(self.copies_in)
        if self.prologue is not None:
            self.prologue()
        fork = None
        if self.branches:
            fork = torch.cuda.Event()
            fork.record(main)
        self.step(**self.kwargs)
        self._copies(self.copies_out)
        for br, st in zip(self.branches, self._streams):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                self._copies(br.copies_in)
                br.step(**br.kwargs)
                self._copies(br.copies_out)
            main.wait_stream(st)

    def replay(self):
        self.graph.replay()


def packed_views(specs, buffer):
    """Views of one byte ``buffer`` for ``specs`` = [(name, shape, dtype), ...], each
    starting on a 256-byte boundary; returns (views dict, bytes used)."""
    views, off = {}, 0
    for name, shape, dtype in specs:
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        views[name] = buffer[off:off + nbytes].view(dtype).view(shape)
        off += (nbytes + 255) // 256 * 256
    return views, off


def packed_size(specs):
    total = 0
    for _, shape, dtype in specs:
        n = 1
        for x in shape:
            n *= x
        total += (n * torch.empty((), dtype=dtype).element_size() + 255) // 256 * 256
    return total
