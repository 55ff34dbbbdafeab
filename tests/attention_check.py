"""Comparison rule of the fused-attention tests (CPU and GPU).

The kernel rounds the softmax probabilities P to the element type before the
P.V product and rounds O once.  With the oracle's fp64 result O and its
weights W = sum_j p_j |v_j| / l and A = sum_j vis_j |v_j| / l (per output
element, ``oracle.attention.attention(..., want_bounds=True)``):
  * rounding each p to a relative error u moves O by at most u W;
  * rounding O moves it by at most u |O|;
  * u = 2^-8 for bf16 (8 significant bits), 2^-11 for fp16 (11 bits);
  * fp16 represents p below 2^-14 as a subnormal, with an absolute error of
    at most 2^-25 each: at most 2^-25 A in all (bf16 has fp32's exponent
    range, and the fp32 exponentials flush only below 2^-126);
  * everything else -- fp32 sums of up to 2^10 partial terms, the SFU
    exponential's ~2^-22 relative error, the fp32 softmax scale, a rotated
    q or k element one unit off where the rotation's fp32 arithmetic and the
    oracle's fp64 one round a near-tie differently -- stays below 2^-14
    (W + |O|).
So |o - O| <= (u + 2^-14)(W + |O|) + s A, s = 2^-25 for fp16 and 0 for bf16.
"""
from __future__ import annotations

import numpy as np

U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
ARITH = 2.0 ** -14
SUBNORMAL = {"bf16": 0.0, "f16": 2.0 ** -25}

# worst err / tol seen per test (printed at the end of the session)
WORST = {}


def tolerance(dtype: str, ref: np.ndarray, w: np.ndarray, a: np.ndarray) -> np.ndarray:
    return (U[dtype] + ARITH) * (w + np.abs(ref)) + SUBNORMAL[dtype] * a


def check(got, ref, w, a, dtype: str, what: str = "") -> float:
    """Assert got (any array of the outputs) within the rule; returns the
    worst err / tol."""
    g = np.asarray(got, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    tol = tolerance(dtype, ref, w, a)
    err = np.abs(g - ref)
    zero_tol = tol == 0
    assert np.all(err[zero_tol] == 0), "%s: %d exact outputs differ" % (
        what, np.count_nonzero(err[zero_tol]))
    ratio = float(np.max(err[~zero_tol] / tol[~zero_tol], initial=0.0))
    bad = np.count_nonzero(err > tol)
    assert bad == 0, "%s: %d of %d beyond tolerance, worst err/tol %.3g, max err %.3g" % (
        what, bad, err.size, ratio, err.max())
    key = what.split(":")[0][:100] or "attention"
    WORST[key] = max(WORST.get(key, 0.0), ratio)
    return ratio


def rejects(got, ref, w, a, dtype: str) -> bool:
    """True when the rule rejects got."""
    try:
        check(got, ref, w, a, dtype, "probe")
    except AssertionError:
        return True
    finally:
        WORST.pop("probe", None)
    return False
