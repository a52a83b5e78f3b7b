"""The pair-score loop evaluates erfc(x) as 2^p(x) with a fitted degree-5
polynomial (csrc/repr.cu).  Its constants must be the fit's, and the error
that reaches a score, |x (erfc(x) - 2^p(x))| per term, must stay below 1e-6
for every x >= 0 in fp32 (it enters each score through at most 256 terms of
|w'| < 0.2, far inside the 2e-3 score tolerance)."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def kernel_coeffs():
    src = open(os.path.join(ROOT, "draft_correction_slot_gb300", "csrc", "repr.cu")).read()
    found = dict(re.findall(r"kErfc(\d) = (-?[0-9.e+-]+)f", src))
    return [float(found[str(k)]) for k in range(6)]


def test_kernel_polynomial_error_bound():
    pytest.importorskip("scipy")
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "fit_erfc", os.path.join(ROOT, "draft_correction_slot_gb300", "fit_erfc.py"))
    fit_erfc = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit_erfc)
    c = kernel_coeffs()
    err, _ = fit_erfc.max_error(c, x_max=12.0)
    assert err < 1e-6
    # far beyond the fitted range 2^p underflows to 0 like erfc
    x = np.float32(30.0)
    p = np.float32(0.0)
    for v in reversed(c):
        p = np.float32(p * x + np.float32(v))
    assert np.exp2(np.float64(p)) == 0.0
    # the constants are those the committed fit produces
    np.testing.assert_allclose(c, fit_erfc.fit(), rtol=1e-6, atol=1e-9)
