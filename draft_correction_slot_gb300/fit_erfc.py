"""Fits the polynomial p with erfc(x) ~ 2^p(x) used by the pair-score loop
(csrc/repr.cu, kErfc0..kErfc5) and reports its error.

The loop evaluates w' |x| erf(|x|) = w' |x| (1 - erfc(|x|)), so the error
that reaches a score is |x| |erfc(x) - 2^p(x)| per term.  p is fitted to
log2 erfc on [0, 5] by weighted least squares, the weights re-scaled each
round by that error (Lawson's iteration towards the smallest maximum), then
checked in fp32 Horner evaluation on [0, 12].  Run it to print the
coefficients and the bound: `python draft_correction_slot_gb300/fit_erfc.py`.
"""
from __future__ import annotations

import numpy as np


def fit(degree: int = 5, x_max: float = 5.0, rounds: int = 60) -> np.ndarray:
    from scipy.special import erfc
    xs = np.linspace(0.0, x_max, 20001)
    target = np.log2(erfc(xs))
    A = np.vander(xs, degree + 1, increasing=True)
    w = np.ones_like(xs)
    c = None
    for _ in range(rounds):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], target * sw, rcond=None)
        err = np.abs(xs * (erfc(xs) - 2.0 ** (A @ c)))
        w = w * (err / err.max() + 1e-3) ** 0.5
        w /= w.mean()
    return c


def max_error(coeffs, x_max: float = 12.0, n: int = 200001) -> tuple[float, float]:
    """max over x in [0, x_max] of |x (erfc(x) - 2^p(x))|, p evaluated in fp32 by Horner."""
    from scipy.special import erfc
    x = np.linspace(0.0, x_max, n).astype(np.float32)
    cf = np.asarray(coeffs, np.float32)
    p = np.full_like(x, cf[-1])
    for k in range(len(cf) - 2, -1, -1):
        p = (p * x + cf[k]).astype(np.float32)
    xd = x.astype(np.float64)
    err = np.abs(xd * (erfc(xd) - np.exp2(p.astype(np.float64))))
    i = int(err.argmax())
    return float(err[i]), float(x[i])


if __name__ == "__main__":
    c = fit()
    e, at = max_error(c)
    print("coefficients (x^0 .. x^5):", ", ".join("%.9g" % v for v in c))
    print("max |x (erfc(x) - 2^p(x))| on [0, 12], fp32: %.3e at x = %.3f" % (e, at))
