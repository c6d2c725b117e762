"""CPU oracle of the fused decode-step sampler (test infrastructure only).

Plain float64 numpy statements of what the sampling side of a decode step
computes, from the fusedtok 1.0.1 README: "Operators" (repetition penalty,
CTRL-style, applied to the ids already sampled; temperature; argmax for greedy
decoding; sample_topp = softmax -> top-p -> seeded draw with a global-mass
threshold; sample_topk = softmax -> top-k -> renormalise within the k survivors ->
seeded draw; decode_step = penalty -> temperature -> nucleus sample in one call,
top-k / top-p with deterministic ties) and "Usage" (the call shapes
``decode_step(logits, sampled_ids, penalty, p, temperature, seed)``,
``sample_topk(logits, k, temperature, seed)``). Shares no code with the CUDA path.

Readings taken where the pages are silent (each is listed in the design notes):
* Repetition penalty (CTRL): every distinct id in ``sampled_ids`` inside [0, V) has
  its logit divided by ``penalty`` when positive and multiplied by it otherwise,
  once however often the id repeats; negative ids are padding.
* Temperature <= 0 means greedy: the argmax of the penalised logits, ties to the
  lowest token id. Otherwise the logits are divided by the temperature and
  softmaxed.
* Ranking: tokens ordered by probability, highest first, equal probabilities by
  token id, lowest first (the deterministic ties).
* top-k (k > 0): the first k tokens of the ranking; k = 0 or k >= V keeps all.
  top-p: within the survivors, renormalised, the shortest prefix of the ranking
  whose mass reaches p (mass >= p); p >= 1 keeps all survivors.
* The draw: the uniform ``u`` in [0, 1) is an input (the random number the method
  draws); the nucleus members are taken in token-id order and the token is the
  first member whose running mass exceeds u times the nucleus mass (inverse CDF in
  id order; the distribution is the renormalised nucleus whatever the order).
"""
from __future__ import annotations

import numpy as np


def repetition_penalty(logits, sampled_ids, penalty):
    """CTRL-style penalty on the distinct ids in [0, V) (fusedtok README, "Operators")."""
    z = np.array(logits, dtype=np.float64)
    V = z.shape[-1]
    ids = {int(i) for i in np.asarray(sampled_ids).ravel() if 0 <= int(i) < V}
    for i in sorted(ids):
        z[i] = z[i] / penalty if z[i] > 0 else z[i] * penalty
    return z


def softmax(z):
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - np.max(z))
    return e / e.sum()


def ranking(p):
    """Token ids by probability, highest first, ties by lowest id."""
    p = np.asarray(p, dtype=np.float64)
    return np.lexsort((np.arange(p.size), -p))


def nucleus(p, top_k=0, top_p=1.0):
    """Boolean mask of the tokens kept by top-k then top-p (readings above)."""
    p = np.asarray(p, dtype=np.float64)
    V = p.size
    order = ranking(p)
    keep = np.zeros(V, dtype=bool)
    n = V if (top_k <= 0 or top_k >= V) else int(top_k)
    kept = order[:n]
    if top_p < 1.0:
        q = p[kept] / p[kept].sum()
        c = np.cumsum(q)
        # shortest prefix whose mass reaches top_p
        m = int(np.searchsorted(c, top_p, side="left")) + 1
        kept = kept[:min(m, n)]
    keep[kept] = True
    return keep


def draw(p, keep, u):
    """First member (in token-id order) whose running mass exceeds u * nucleus mass."""
    p = np.asarray(p, dtype=np.float64)
    idx = np.nonzero(keep)[0]
    c = np.cumsum(p[idx])
    t = u * c[-1]
    j = int(np.searchsorted(c, t, side="right"))
    return int(idx[min(j, idx.size - 1)])


def sample(logits, sampled_ids, penalty=1.0, temperature=1.0, top_p=1.0, top_k=0, u=0.0):
    """decode_step of the sampling side for one row: penalty -> temperature ->
    (argmax | softmax -> top-k -> top-p -> draw). Returns the token id."""
    z = repetition_penalty(logits, sampled_ids, penalty)
    if temperature <= 0:
        return int(np.argmax(z))  # first maximum: lowest id among ties
    p = softmax(z / temperature)
    return draw(p, nucleus(p, top_k, top_p), u)


def decision_margins(logits, sampled_ids, penalty=1.0, temperature=1.0, top_p=1.0, top_k=0,
                     u=0.0):
    """How far the two real-valued decisions of :func:`sample` are from a boundary,
    as fractions of the total mass: the top-p cut (the nucleus mass before and after
    its last member against p) and the draw (the target against the running masses
    of the chosen member and its predecessor). A GPU sampler working in fp32 may only
    disagree with this fp64 oracle when one of them is tiny."""
    z = repetition_penalty(logits, sampled_ids, penalty)
    if temperature <= 0:
        s = np.sort(z)[::-1]
        return {"argmax_gap": float(s[0] - s[1]) if s.size > 1 else np.inf}
    p = softmax(z / temperature)
    V = p.size
    order = ranking(p)
    n = V if (top_k <= 0 or top_k >= V) else int(top_k)
    kept = order[:n]
    cut = np.inf
    if top_p < 1.0:
        q = p[kept] / p[kept].sum()
        c = np.cumsum(q)
        m = int(np.searchsorted(c, top_p, side="left"))
        before = c[m - 1] if m > 0 else 0.0
        cut = float(min(abs(c[min(m, n - 1)] - top_p), abs(top_p - before)))
    keep = nucleus(p, top_k, top_p)
    idx = np.nonzero(keep)[0]
    c = np.cumsum(p[idx]) / p[idx].sum()
    j = int(np.searchsorted(c, u, side="right"))
    j = min(j, idx.size - 1)
    lo = c[j - 1] if j > 0 else 0.0
    return {"top_p_cut": cut, "draw": float(min(abs(c[j] - u), abs(u - lo)))}
