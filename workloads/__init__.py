"""Seeded synthetic inputs for the decode-step attention block.

This module is shared by the tests, the benchmark and the smoke check. It only
draws random numbers and lays them out; it holds none of the block's arithmetic
(no norm, no rotation, no softmax). Both the CUDA path and the CPU oracle consume
exactly the bf16 bit patterns produced here.

Recipe (one numpy ``Generator(PCG64(seed))`` per call, draws in this order):

1. ``lens``   per-sequence context length after the append (int32, [B]);
2. ``x``      new hidden state          [B, hidden]   ~ N(0, 1);
3. ``residual`` residual stream         [B, hidden]   ~ N(0, residual_var);
4. ``norm_w`` RMSNorm weight            [hidden]      = 1 + 0.1 N(0, 1);
5. ``q``      new-token queries         [B, Hq, D]    ~ N(0, 1);
6. ``k_new``  new-token keys            [B, Hkv, D]   ~ N(0, 1);
7. ``v_new``  new-token values          [B, Hkv, D]   ~ N(0, 1);
8. ``q_norm_w``, ``k_norm_w`` per-head norm weights [D] = 1 + 0.1 N(0, 1)
   (drawn only when QK-norm is on);
9. for each sequence b: the K cache prefix [Hkv, pos_b, D] then the V cache
   prefix [Hkv, pos_b, D], ~ N(0, 1);
10. key spikes (long-context case): a set of cache positions, drawn without
    replacement, whose keys are multiplied by a power of two (exact in bf16).

Every float draw is float32, rounded to bf16 with round-to-nearest-even by
``torch.Tensor.to(torch.bfloat16)``. Cache slots past ``pos_b`` (and every slot of
an unused capacity tail) hold the bf16 quiet-NaN sentinel, so a kernel that reads
outside the valid range poisons its output. ``pos_b = lens_b - 1``: the new token
is written at slot ``pos_b`` and is the last of the ``lens_b`` tokens attended.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

NEOX = "neox"
INTERLEAVED = "interleaved"


@dataclasses.dataclass(frozen=True)
class BlockConfig:
    """Shape and value recipe of one decode-step attention workload."""

    name: str
    B: int
    hidden: int
    Hq: int
    Hkv: int
    D: int
    theta: float
    layout: str
    qk_norm: bool
    lens_kind: str              # "fixed", "uniform", "geometric"
    lens_args: tuple
    residual_var: float = 1.0
    eps: float = 1e-6
    key_spike_frac: float = 0.0
    key_spike_scale: float = 1.0
    t_cap: int | None = None    # None: the largest length in the batch
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def replace(self, **kw) -> "BlockConfig":
        return dataclasses.replace(self, **kw)


# The five workloads of the decode-step attention block, sizes as the pages'
# models (Qwen3-0.6B, Llama-3-8B) and serving regimes shape them.
TINY = BlockConfig("tiny", B=1, hidden=256, Hq=4, Hkv=1, D=64, theta=1e4,
                   layout=NEOX, qk_norm=False, lens_kind="fixed", lens_args=(128,))
QWEN3_128 = BlockConfig("qwen3_0p6b_ctx128", B=1, hidden=1024, Hq=16, Hkv=8, D=128,
                        theta=1e6, layout=NEOX, qk_norm=True, lens_kind="fixed",
                        lens_args=(128,), residual_var=4.0)
QWEN3_512 = QWEN3_128.replace(name="qwen3_0p6b_ctx512", lens_args=(512,))
LLAMA3_BATCHED = BlockConfig("llama3_8b_batched", B=32, hidden=4096, Hq=32, Hkv=8, D=128,
                             theta=5e5, layout=NEOX, qk_norm=False, lens_kind="uniform",
                             lens_args=(512, 8192), t_cap=8192)
LONG_CONTEXT = BlockConfig("long_context_131k", B=1, hidden=4096, Hq=32, Hkv=8, D=128,
                           theta=5e5, layout=NEOX, qk_norm=False, lens_kind="fixed",
                           lens_args=(131072,), key_spike_frac=0.01, key_spike_scale=8.0)
SERVING_MIX = BlockConfig("serving_mix", B=256, hidden=2048, Hq=16, Hkv=4, D=128,
                          theta=1e4, layout=INTERLEAVED, qk_norm=True, lens_kind="geometric",
                          lens_args=(2048, 32768))

CONFIGS = {c.name: c for c in (TINY, QWEN3_128, QWEN3_512, LLAMA3_BATCHED, LONG_CONTEXT,
                               SERVING_MIX)}

BF16_NAN_BITS = 0x7FC0


def draw_lens(cfg: BlockConfig, rng: np.random.Generator) -> np.ndarray:
    """Per-sequence lengths (after the new token is appended)."""
    if cfg.lens_kind == "fixed":
        lens = np.full(cfg.B, int(cfg.lens_args[0]), dtype=np.int64)
    elif cfg.lens_kind == "uniform":
        lo, hi = cfg.lens_args
        lens = rng.integers(lo, hi, size=cfg.B, endpoint=True)
    elif cfg.lens_kind == "geometric":
        mean, cap = cfg.lens_args
        lens = np.minimum(rng.geometric(1.0 / mean, size=cfg.B), cap)
    elif cfg.lens_kind == "list":
        lens = np.asarray(cfg.lens_args, dtype=np.int64)
        assert lens.shape == (cfg.B,)
    else:
        raise ValueError(cfg.lens_kind)
    return lens.astype(np.int32)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng, shape, std=1.0, mean=0.0):
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return a


def nan_bf16(shape) -> torch.Tensor:
    return torch.full(shape, BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16)


def make_inputs(cfg: BlockConfig, with_cache: bool = True) -> dict:
    """Draw one decode step's inputs for ``cfg`` (CPU tensors, bf16 / int32)."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    lens = draw_lens(cfg, rng)
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    t_cap = int(cfg.t_cap if cfg.t_cap is not None else max(int(lens.max(initial=1)), 1))
    if lens.size and int(lens.max()) > t_cap:
        raise ValueError("a length exceeds the cache capacity")
    out = {"cfg": cfg, "t_cap": t_cap, "lens": torch.from_numpy(lens.copy()),
           "pos": torch.from_numpy(np.maximum(lens - 1, 0).astype(np.int32))}
    out["x"] = _bf16(_normal(rng, (B, H)))
    out["residual"] = _bf16(_normal(rng, (B, H), std=math.sqrt(cfg.residual_var)))
    out["norm_w"] = _bf16(_normal(rng, (H,), std=0.1, mean=1.0))
    out["q"] = _bf16(_normal(rng, (B, Hq, D)))
    out["k_new"] = _bf16(_normal(rng, (B, Hkv, D)))
    out["v_new"] = _bf16(_normal(rng, (B, Hkv, D)))
    if cfg.qk_norm:
        out["q_norm_w"] = _bf16(_normal(rng, (D,), std=0.1, mean=1.0))
        out["k_norm_w"] = _bf16(_normal(rng, (D,), std=0.1, mean=1.0))
    else:
        out["q_norm_w"] = None
        out["k_norm_w"] = None
    if not with_cache:
        return out
    k_cache = nan_bf16((B, Hkv, t_cap, D))
    v_cache = nan_bf16((B, Hkv, t_cap, D))
    for b in range(B):
        n = int(lens[b]) - 1           # tokens already in the cache before the append
        if n <= 0:
            continue
        k_cache[b, :, :n] = _bf16(_normal(rng, (Hkv, n, D)))
        v_cache[b, :, :n] = _bf16(_normal(rng, (Hkv, n, D)))
    if cfg.key_spike_frac > 0.0:
        for b in range(B):
            n = int(lens[b]) - 1
            cnt = int(round(cfg.key_spike_frac * n))
            if cnt <= 0:
                continue
            where = np.sort(rng.choice(n, size=cnt, replace=False))
            idx = torch.from_numpy(where.astype(np.int64))
            k_cache[b, :, idx] = k_cache[b, :, idx] * cfg.key_spike_scale
    out["k_cache"] = k_cache
    out["v_cache"] = v_cache
    return out


def small_variant(cfg: BlockConfig, B: int | None = None, max_len: int | None = None,
                  seed: int | None = None) -> BlockConfig:
    """The same recipe at a size the CPU oracle finishes in seconds.

    Lengths keep their distribution family, clipped to ``max_len``.
    """
    kw = {}
    if B is not None:
        kw["B"] = B
    if seed is not None:
        kw["seed"] = seed
    if max_len is not None:
        if cfg.lens_kind == "fixed":
            kw["lens_args"] = (min(cfg.lens_args[0], max_len),)
        elif cfg.lens_kind == "uniform":
            lo, hi = cfg.lens_args
            kw["lens_args"] = (min(lo, max_len // 4), max_len)
        elif cfg.lens_kind == "geometric":
            mean, cap = cfg.lens_args
            kw["lens_args"] = (max(1, min(mean, max_len // 4)), max_len)
        kw["t_cap"] = None
    return cfg.replace(name=cfg.name + "_small", **kw)


def algorithmic_bytes(cfg: BlockConfig, lens, num_partials: int = 0) -> dict:
    """Bytes one decode step must move at minimum, per kernel.

    KV stream: every attended K and V row once. RMSNorm: read x, residual, weight,
    write y and the new residual. Append: read and write q, read k_new/v_new (and
    the two norm weights when QK-norm is on), write the K and V slots. Attention:
    the KV stream, q and the lengths in, the output out. The split-KV partials are
    an artefact of this implementation, not of the method, so they are not counted
    (``partials`` reports them for ``num_partials`` partial slots).
    """
    lens = np.asarray(lens, dtype=np.int64)
    B, H, Hq, Hkv, D, G = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D, cfg.G
    tokens = int(lens.sum())
    kv = 2 * Hkv * D * 2 * tokens
    rms = (4 * B * H + H) * 2
    append = (2 * B * Hq * D + 2 * B * Hkv * D + 2 * B * Hkv * D) * 2 + B * 4
    if cfg.qk_norm:
        append += 2 * D * 2
    attn_split = kv + B * Hq * D * 2 + B * 4
    merge = B * Hq * D * 2
    return {"rmsnorm": rms, "append": append, "attn_split": attn_split, "merge": merge,
            "attn": attn_split + merge, "kv": kv, "step": rms + append + attn_split + merge,
            "partials": num_partials * G * (D + 1) * 4}


# ------------------------------------------------ projections around the block ---
PROJ_SEED_OFFSET = 7919  # projection weights draw from their own stream


def make_projection_weights(cfg: BlockConfig) -> dict:
    """Weights of the packed QKV and output projections, random-init, bf16.

    One ``Generator(PCG64(cfg.seed + PROJ_SEED_OFFSET))``, draws in this order:
    ``w_qkv`` [(Hq + 2 Hkv) D, hidden] ~ N(0, 1/hidden), then ``w_o`` [hidden, Hq D]
    ~ N(0, 1/(Hq D)) (rows = output features; the fan-in scaling keeps the
    projected values of order one)."""
    rng = np.random.default_rng(cfg.seed + PROJ_SEED_OFFSET)
    nqkv = (cfg.Hq + 2 * cfg.Hkv) * cfg.D
    w_qkv = _bf16(_normal(rng, (nqkv, cfg.hidden), std=1.0 / math.sqrt(cfg.hidden)))
    w_o = _bf16(_normal(rng, (cfg.hidden, cfg.Hq * cfg.D), std=1.0 / math.sqrt(cfg.Hq * cfg.D)))
    return {"w_qkv": w_qkv, "w_o": w_o}


def make_linear_inputs(B: int, N: int, K: int, seed: int = 0, residual: bool = True) -> dict:
    """x [B, K] ~ N(0, 1), w [N, K] ~ N(0, 1/K), residual [B, N] ~ N(0, 1), bf16, drawn in
    that order from ``Generator(PCG64(seed))``."""
    rng = np.random.default_rng(seed)
    out = {"x": _bf16(_normal(rng, (B, K))),
           "w": _bf16(_normal(rng, (N, K), std=1.0 / math.sqrt(K)))}
    out["residual"] = _bf16(_normal(rng, (B, N))) if residual else None
    return out


def make_norm_linear_inputs(B: int, N: int, K: int, seed: int = 0,
                            residual: bool = True) -> dict:
    """Inputs of a projection with the RMSNorm prologue: x [B, K] ~ N(0, 1), w [N, K] ~
    N(0, 1/K), norm_w [K] = 1 + 0.1 N(0, 1), residual [B, K] ~ N(0, 4), bf16, drawn in
    that order from ``Generator(PCG64(seed))``."""
    rng = np.random.default_rng(seed)
    out = {"x": _bf16(_normal(rng, (B, K))),
           "w": _bf16(_normal(rng, (N, K), std=1.0 / math.sqrt(K))),
           "norm_w": _bf16(1.0 + 0.1 * _normal(rng, (K,)))}
    out["residual"] = _bf16(_normal(rng, (B, K), std=2.0)) if residual else None
    return out


def sublayer_bytes(cfg: BlockConfig, lens) -> dict:
    """Bytes the attention sublayer must move at minimum: the block's, with q, k_new
    and v_new produced by the QKV projection instead of read as inputs, plus both
    weights once, the projections' activations and the output (read h, write out)."""
    blk = algorithmic_bytes(cfg, lens)
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    nqkv = (Hq + 2 * Hkv) * D
    qkv_proj = (nqkv * H + B * H + B * nqkv) * 2
    o_proj = (H * Hq * D + B * Hq * D + 2 * B * H) * 2
    return {"rmsnorm": blk["rmsnorm"], "qkv_proj": qkv_proj, "append": blk["append"],
            "attn": blk["attn_split"] + blk["merge"], "o_proj": o_proj, "block": blk["step"],
            "weights": (nqkv * H + H * Hq * D) * 2, "kv": blk["kv"],
            "step": blk["step"] + qkv_proj + o_proj}


def linear_flops(B: int, N: int, K: int) -> int:
    return 2 * B * N * K


# ---------------------------------------------------------------- sampler ---
SAMPLER_VOCAB = 131072  # the pages' sampler benchmarks run on rows of 131072 logits


def make_sampler_inputs(B: int, V: int, kind: str = "peaked", L: int = 64, seed: int = 0) -> dict:
    """Rows of fp32 logits, previously sampled ids and uniforms, drawn in that order from
    ``Generator(PCG64(seed))``.

    kind: ``peaked`` N(0, 2^2) plus +8 on 1% of the ids (decode-like: a few likely
    tokens); ``flat`` N(0, 0.05^2) (the nucleus spans most of the row); ``ties``
    integers in [-3, 3] (many exactly equal logits); ``masked`` peaked with 30% of the
    ids at -inf. ids: L per row, uniform over [-2, V + 2) (negative = padding, >= V
    ignored), duplicates allowed. u: uniform in [0, 1), float32.
    """
    rng = np.random.default_rng(seed)
    if kind == "flat":
        z = rng.standard_normal((B, V), dtype=np.float32) * np.float32(0.05)
    elif kind == "ties":
        z = rng.integers(-3, 4, size=(B, V)).astype(np.float32)
    else:
        z = rng.standard_normal((B, V), dtype=np.float32) * np.float32(2.0)
        spikes = rng.random((B, V)) < 0.01
        z = np.where(spikes, z + np.float32(8.0), z).astype(np.float32)
        if kind == "masked":
            z = np.where(rng.random((B, V)) < 0.3, np.float32(-np.inf), z).astype(np.float32)
    ids = rng.integers(-2, V + 2, size=(B, L)).astype(np.int32)
    u = rng.random(B, dtype=np.float32)
    return {"logits": torch.from_numpy(np.ascontiguousarray(z)),
            "ids": torch.from_numpy(ids), "u": torch.from_numpy(u)}
