"""The fused sampler (CUDA) against the CPU oracle on identical seeded rows (GPU only).

The token is an integer decided by real-valued comparisons. The GPU takes them in
fp32 exponentials and 2^-40 fixed-point masses, the oracle in fp64, so the tokens
must match exactly whenever the oracle's decisions are not within 1e-5 (relative
mass) of a boundary; inside that band either neighbouring outcome is accepted,
found by re-running the oracle with u and top_p moved by the band.
"""
import numpy as np
import pytest
import torch

import decode_step_attention_gb300 as dsa
import workloads as W
from oracle import sampler as S

pytestmark = pytest.mark.gpu

DEV = "cuda"
BAND = 1e-5

PARAMS = [  # penalty, temperature, top_p, top_k
    (1.0, 0.0, 1.0, 0),     # greedy
    (1.3, 0.0, 1.0, 0),     # greedy after the penalty
    (1.1, 0.8, 0.9, 0),     # decode_step of the pages' usage
    (1.0, 1.0, 1.0, 0),     # plain softmax draw
    (1.0, 0.8, 1.0, 50),    # sample_topk of the pages' usage
    (1.2, 1.0, 0.5, 10),    # top-k then top-p
    (2.0, 1.5, 0.95, 1),    # top-k = 1 is greedy over the tempered row
    (1.0, 0.7, 0.999, 0),
]


def _accepted(z, ids, pen, T, p, k, u):
    tok = S.sample(z, ids, pen, T, p, k, u)
    m = S.decision_margins(z, ids, pen, T, p, k, u)
    if min(m.values()) >= BAND:
        return {tok}
    ok = {tok}
    for du in (-BAND, 0.0, BAND):
        for dp in ((-BAND, 0.0, BAND) if p < 1.0 else (0.0,)):
            uu = min(max(u + du, 0.0), np.nextafter(1.0, 0.0))
            ok.add(S.sample(z, ids, pen, T, min(p + dp, 1.0), k, uu))
    return ok


def _check(inp, pen, T, p, k, what):
    z, ids, u = inp["logits"], inp["ids"], inp["u"]
    tok = dsa.sample(z.to(DEV), ids.to(DEV), pen, T, p, k, u=u.to(DEV)).cpu().numpy()
    zz, ii, uu = z.double().numpy(), ids.numpy(), u.double().numpy()
    for b in range(z.shape[0]):
        acc = _accepted(zz[b], ii[b], pen, T, p, k, float(uu[b]))
        assert int(tok[b]) in acc, (what, b, int(tok[b]), acc)


@pytest.mark.parametrize("V", [7, 1000, 4096, 4097, 32000, 65537, 131072, 151936, 262144])
@pytest.mark.parametrize("params", PARAMS)
def test_sampler_matches_oracle(V, params):
    inp = W.make_sampler_inputs(4, V, "peaked", L=32, seed=V % 1000)
    _check(inp, *params, f"V={V} {params}")


@pytest.mark.parametrize("kind", ["flat", "ties", "masked"])
@pytest.mark.parametrize("params", PARAMS)
def test_sampler_distributions(kind, params):
    inp = W.make_sampler_inputs(3, 50021, kind, L=200, seed=7)
    _check(inp, *params, f"{kind} {params}")


def test_sampler_many_rows_and_uniforms():
    """64 rows of the pages' vocabulary size, each with its own u."""
    inp = W.make_sampler_inputs(64, W.SAMPLER_VOCAB, "peaked", L=128, seed=3)
    _check(inp, 1.1, 0.8, 0.9, 0, "batch")


def test_sampler_u_grid_small_vocab():
    """One row, u on a grid: the GPU's token for every u equals the oracle's (the draw
    maps the unit interval onto the nucleus in token-id order)."""
    base = W.make_sampler_inputs(1, 40, "peaked", L=5, seed=11)
    n = 400
    z = base["logits"].repeat(n, 1)
    ids = base["ids"].repeat(n, 1)
    u = ((torch.arange(n, dtype=torch.float64) + 0.5) / n).float()
    _check({"logits": z, "ids": ids, "u": u}, 1.2, 0.9, 0.85, 12, "u grid")


def test_sampler_repeatable_and_special_cases():
    inp = W.make_sampler_inputs(8, 20000, "ties", L=16, seed=5)
    z, ids, u = inp["logits"].to(DEV), inp["ids"].to(DEV), inp["u"].to(DEV)
    a = dsa.sample(z, ids, 1.1, 0.9, 0.9, 0, u=u)
    b = dsa.sample(z, ids, 1.1, 0.9, 0.9, 0, u=u)
    assert torch.equal(a, b)
    # top_k = 1 and a tiny top_p both give the argmax of the penalised row
    g = dsa.sample(z, ids, 1.1, 0.0)
    assert torch.equal(dsa.sample(z, ids, 1.1, 0.9, 1.0, 1, u=u), g)
    assert torch.equal(dsa.sample(z, ids, 1.1, 0.9, 1e-6, 0, u=u), g)
    # no ids, seeded uniforms through the binding
    t1 = dsa.sample(z, None, 1.0, 1.0, 0.9, 0, seed=123)
    t2 = dsa.sample(z, None, 1.0, 1.0, 0.9, 0, seed=123)
    assert torch.equal(t1, t2)
    # empty batch
    e = dsa.sample(torch.empty(0, 100, device=DEV), None, 1.0, 1.0)
    assert e.shape == (0,)


@pytest.mark.parametrize("kind", ["peaked", "flat", "ties", "masked"])
@pytest.mark.parametrize("params", PARAMS)
def test_sampler_batch_independent(kind, params):
    """A batch large enough to change the cluster size: parity with the oracle on
    sampled rows, and the same tokens as the same rows sampled 8 at a time (the same
    operations give the same e, and every sum is an integer sum)."""
    B = 160
    inp = W.make_sampler_inputs(B, 32768, kind, L=64, seed=17)
    z, ids, u = inp["logits"].to(DEV), inp["ids"].to(DEV), inp["u"].to(DEV)
    big = dsa.sample(z, ids, *params, u=u)
    small = torch.cat([dsa.sample(z[i:i + 8], ids[i:i + 8], *params, u=u[i:i + 8])
                       for i in range(0, B, 8)])
    assert torch.equal(big, small)
    rows = list(range(0, B, 23))
    sub = {k: v[rows] for k, v in inp.items()}
    _check(sub, *params, f"batch {kind} {params}")


@pytest.mark.parametrize("kind", ["peaked", "flat", "ties", "masked"])
@pytest.mark.parametrize("top_k", [2, 50, 700, 2048, 2049, 5000])
def test_sampler_top_k_then_top_p(kind, top_k):
    """Top-k then top-p on both sides of the 2048-survivor limit below which the top-p
    select runs on the survivors alone (ties across the cut in the "ties" rows)."""
    inp = W.make_sampler_inputs(6, 65536, kind, L=40, seed=top_k)
    for p in (0.3, 0.9, 0.999):
        _check(inp, 1.1, 0.9, p, top_k, f"{kind} top_k={top_k} top_p={p}")
