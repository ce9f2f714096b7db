"""Comparison rules shared by the GPU parity tests.

Tolerances (bf16 inputs, fp32 accumulation, fp64 oracle):
  O   : max |O - O_ref| <= 1e-2 beyond the output format's own rounding.  O is
        stored in bf16, whose rounding alone reaches 2^-8 |O| (half an ulp),
        which exceeds 1e-2 once |O| > 2.56; the check therefore bounds
        |O - O_ref| - 2^-8 |O_ref|.  The raw maximum is reported as well.
  lse : max |lse - lse_ref| <= 1e-3 (lse is fp32).
  dQ, dK, dV : relative Frobenius error <= 2e-2 (denominator floored at an
        RMS of 1e-4 per element, for gradients that are exactly zero).
"""
import numpy as np

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_TOL = 2e-2
BF16_HALF_ULP_REL = 2.0 ** -8


def o_excess(o_gpu, o_ref):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    diff = np.abs(o_gpu - o_ref)
    return float(np.max(diff - BF16_HALF_ULP_REL * np.abs(o_ref))), float(np.max(diff))


def assert_o(o_gpu, o_ref, what=""):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    excess, raw = o_excess(o_gpu, o_ref)
    assert excess <= O_TOL, f"{what}: |dO| beyond bf16 rounding {excess:.3e} (raw {raw:.3e})"
    return raw


def assert_lse(l_gpu, l_ref, what=""):
    l_gpu = np.asarray(l_gpu, np.float64)
    l_ref = np.asarray(l_ref, np.float64)
    both_inf = np.isneginf(l_gpu) & np.isneginf(l_ref)
    err = np.where(both_inf, 0.0, np.abs(l_gpu - l_ref))
    m = float(np.max(err)) if err.size else 0.0
    assert m <= LSE_TOL, f"{what}: |dlse| {m:.3e}"
    return m


# Floor of the relative-error denominator: an RMS of 1e-4 per element.  It only
# matters where the exact gradient vanishes (a softmax over a single key has
# zero gradient with respect to q and k), where a relative error is undefined.
GRAD_RMS_FLOOR = 1e-4


def rel_fro(g, ref):
    g = np.asarray(g, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = GRAD_RMS_FLOOR * np.sqrt(ref.size)
    return float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), floor))


def assert_grad(g, ref, what=""):
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    e = rel_fro(g, ref)
    assert e <= GRAD_TOL, f"{what}: relative Frobenius error {e:.3e}"
    return e
