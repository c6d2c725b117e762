"""The CPU oracle against its pins (closed forms, invariants, special cases,
hand-derived fixtures and scalar brute force). CPU only."""
import numpy as np
import pytest
import torch

import pins
import workloads
import types

from oracle import decode_ref as O
from oracle import sampler as SAMPLER

# the oracle as the pins see it: the block's functions, and the sampler beside them
ORACLE = types.SimpleNamespace(**{k: getattr(O, k) for k in dir(O) if not k.startswith("_")},
                               sampler=SAMPLER)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ORACLE)


def test_generators_reproducible():
    cfg = workloads.small_variant(workloads.SERVING_MIX, B=6, max_len=300)
    a = workloads.make_inputs(cfg)
    b = workloads.make_inputs(cfg)
    for k in ("x", "residual", "q", "k_new", "v_new", "k_cache", "v_cache", "lens", "pos"):
        assert torch.equal(a[k].view(torch.int16) if a[k].dtype == torch.bfloat16 else a[k],
                           b[k].view(torch.int16) if b[k].dtype == torch.bfloat16 else b[k]), k
    c = workloads.make_inputs(cfg.replace(seed=1))
    assert not torch.equal(a["q"], c["q"])


def test_generator_layout():
    cfg = workloads.small_variant(workloads.LLAMA3_BATCHED, B=5, max_len=200)
    inp = workloads.make_inputs(cfg)
    lens = inp["lens"].numpy()
    assert np.all(inp["pos"].numpy() == lens - 1)
    kc = inp["k_cache"].float().numpy()
    for b in range(cfg.B):
        n = lens[b] - 1
        assert np.all(np.isfinite(kc[b, :, :n]))
        assert np.all(np.isnan(kc[b, :, n:]))  # the new slot and the tail are sentinels
    assert inp["q_norm_w"] is None


def test_long_context_spikes():
    cfg = workloads.LONG_CONTEXT.replace(lens_args=(2001,), Hkv=2, Hq=8)
    inp = workloads.make_inputs(cfg)
    kc = inp["k_cache"].float().numpy()[0]
    big = np.abs(kc).max(axis=(0, 2))[:2000]
    assert (big > 8.0).sum() >= 15  # 20 spiked positions, most exceed |x| > 8 after x8


def test_decode_step_composes():
    cfg = workloads.small_variant(workloads.QWEN3_128, max_len=40)
    inp = workloads.make_inputs(cfg)
    f = {k: (v.double().numpy() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    f.update(eps=cfg.eps, theta=cfg.theta, layout=cfg.layout)
    res = O.decode_step(f)
    assert np.all(np.isfinite(res["out"]))
    assert np.all(np.isfinite(res["k_cache"][0, :, :40]))
