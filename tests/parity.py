"""Comparison rules shared by the GPU parity tests.

Tolerances (bf16 inputs, fp32 accumulation, fp64 oracle):
  O   : max |O - O_ref| <= 1e-2 for the value the kernel computed before it
        stored O in bf16.  Only the stored bf16 value is visible, and that
        rounding alone moves a value by up to half a bf16 ulp of its own binade
        (2^(e - 8) for |O| in [2^e, 2^(e+1))), which exceeds 1e-2 once |O| >= 4.
        The check therefore allows exactly that half ulp of the GPU's own value
        on top of 1e-2: |O - O_ref| <= 1e-2 + halfulp_bf16(O).  For |O| < 1 the
        allowance is at most 2^-9; the raw maximum is reported as well.
  lse : max |lse - lse_ref| <= 1e-3 (lse is fp32).
  dQ, dK, dV : relative Frobenius error <= 2e-2 (denominator floored at an
        RMS of 1e-4 per element, for gradients that are exactly zero).
"""
import numpy as np

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_TOL = 2e-2


def bf16_half_ulp(x):
    """Half the spacing of bf16 values (8 significant bits) in the binade of
    each |x|: 2^(floor(log2 |x|) - 8); 0 where x = 0 (bf16 stores 0 exactly)."""
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(x)                      # x = m 2^e with m in [0.5, 1): binade 2^(e-1)
    return np.where(x > 0, np.ldexp(1.0, e - 1 - 8), 0.0)


def bf16_round(x):
    """x rounded to the nearest bf16 value, ties to even, computed exactly in
    float64 (one rounding; no detour through float32)."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                      # |m| in [0.5, 1): 8 significant bits = m * 2^8
    return np.ldexp(np.rint(m * 256.0), e - 8)


def o_excess(o_gpu, o_ref):
    """(max of |O - O_ref| - halfulp_bf16(O), max |O - O_ref|)."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    diff = np.abs(o_gpu - o_ref)
    return float(np.max(diff - bf16_half_ulp(o_gpu))), float(np.max(diff))


def assert_o(o_gpu, o_ref, what=""):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    excess, raw = o_excess(o_gpu, o_ref)
    assert excess <= O_TOL, f"{what}: |dO| beyond the bf16 output rounding {excess:.3e} (raw {raw:.3e})"
    return raw


def assert_lse(l_gpu, l_ref, what=""):
    l_gpu = np.asarray(l_gpu, np.float64)
    l_ref = np.asarray(l_ref, np.float64)
    both_inf = np.isneginf(l_gpu) & np.isneginf(l_ref)
    with np.errstate(invalid="ignore"):
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
