"""The cubic of the software exp2 ("efficient-attention/flash-2-3", section
"And on Blackwell": 2^x = 2^floor(x) * p3(x - floor(x)) evaluated on the FMA
units).  CPU pins, independent of the GPU:

  * the fitting script, re-run here, reproduces the constants compiled into
    the kernels (so the constants are the script's, not copied from anywhere);
  * the fitted cubic's largest relative error against 2^f on [0, 1], computed
    in float64 on a grid ten times denser than the fit's, is the stated
    8.6e-5, and p3(0) = 1 exactly (integer x gives the exact power of two);
  * the error bound discriminates: dropping a term or flipping a sign moves the
    error far beyond it.
"""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_94_gb300", "csrc")
BOUND = 8.6e-5


def compiled_coefficients():
    text = open(os.path.join(CSRC, "ptx.cuh")).read()
    return [float(re.search(rf"kExp2C{i}\s*=\s*([0-9.eE+-]+)f", text).group(1)) for i in (1, 2, 3)]


def fit_script():
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", os.path.join(CSRC, "fit_exp2_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def cubic(c, f):
    return 1.0 + f * (c[0] + f * (c[1] + f * c[2]))


def max_rel_err(c):
    f = np.linspace(0.0, 1.0, 40001)
    return float(np.max(np.abs(cubic(c, f) - np.exp2(f)) / np.exp2(f)))


def test_script_reproduces_the_compiled_constants():
    pytest.importorskip("scipy")
    c_fit, err = fit_script().fit()
    c_hdr = compiled_coefficients()
    assert np.allclose(c_fit, c_hdr, rtol=1e-8, atol=0), (c_fit, c_hdr)
    assert abs(err - BOUND) < 0.05 * BOUND


def test_cubic_error_is_the_stated_bound():
    c = compiled_coefficients()
    e = max_rel_err(c)
    assert 0.95 * BOUND <= e <= 1.01 * BOUND, e
    assert cubic(c, 0.0) == 1.0
    # continuity at f -> 1: p3(1) ~ 2, within the bound, so 2^floor(x) * p3 has no jump at integers
    assert abs(cubic(c, 1.0) / 2.0 - 1.0) <= BOUND * 1.01


@pytest.mark.parametrize("mutate", ["drop_c3", "neg_c2", "swap_c1_c2"])
def test_plausible_mistakes_break_the_bound(mutate):
    c = compiled_coefficients()
    if mutate == "drop_c3":
        c = [c[0], c[1], 0.0]
    elif mutate == "neg_c2":
        c = [c[0], -c[1], c[2]]
    else:
        c = [c[1], c[0], c[2]]
    assert max_rel_err(c) > 100 * BOUND
