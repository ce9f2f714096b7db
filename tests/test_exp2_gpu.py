"""The kernels' software exp2 on the GPU ("efficient-attention/flash-2-3",
section "And on Blackwell": part of the exponentials on the FMA units as
2^floor(x) * p3(x - floor(x))), evaluated through fa_selftest_exp2 on a dense
grid of x and compared with float64 2^x and with CUDA's exp2f.

Bound: the cubic's fitted relative error 8.6e-5 plus the float32 rounding of
the evaluation (the fraction x - floor(x), three fused multiply-adds: a few
float32 ulps, 4e-7 allowed) on x in [-126, 0], where 2^x is a normal float32.
Below -126 the result is tiny (at most 2^-126 in absolute value, inputs
below -127 clamped); there only the absolute size is checked.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_94_gb300 import _lib

pytestmark = pytest.mark.gpu

REL = 8.6e-5 + 4e-7


def run(x, which):
    xt = torch.as_tensor(np.asarray(x, np.float32)).cuda()
    y = torch.empty_like(xt)
    st = _lib.load().fa_selftest_exp2(ctypes.c_void_p(xt.data_ptr()), ctypes.c_void_p(y.data_ptr()), xt.numel(),
                                      which, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.FA_OK
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def grid():
    rng = np.random.default_rng(0)
    dense = np.linspace(-126.0, 0.0, 1 << 21)
    ints = -np.arange(0, 127, dtype=np.float64)
    near_ints = np.concatenate([ints + 1e-6, ints - 1e-6, ints + 0.5])
    rand = -rng.random(1 << 18) * 126.0
    x = np.concatenate([dense, ints, near_ints, rand]).astype(np.float32)
    return x[(x >= -126.0) & (x <= 0.0)]


def test_cubic_against_float64():
    x = grid()
    y = run(x, 0)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() <= REL, float(rel.max())
    assert rel.max() >= 0.5 * 8.6e-5   # it is the cubic (an exact exp would be ~1e-7)
    ints = -np.arange(0, 127, dtype=np.float32)
    assert np.array_equal(run(ints, 0), np.exp2(ints.astype(np.float64)))  # p3(0) = 1: exact powers of two


def test_packed_cubic_is_the_scalar_cubic_bit_for_bit():
    """The forward kernel evaluates the cubic on pairs with the packed f32x2
    instructions; the results must be those of the scalar form exactly."""
    x = np.concatenate([grid(), np.array([-126.5, -127.0, -130.0, -np.inf, 0.0], np.float32)])
    assert np.array_equal(run(x, 3), run(x, 0))
    assert np.array_equal(run(x[:-1], 3), run(x[:-1], 0))  # an odd count: the last value alone


def test_cubic_against_exp2f():
    x = grid()
    y_poly = run(x, 0)
    y_f = run(x, 2)
    rel = np.abs(y_poly - y_f) / y_f
    assert rel.max() <= REL + 3e-7, float(rel.max())   # exp2f is within 2 ulp of 2^x


def test_sfu_exp2_against_float64():
    """The SFU path the kernels use by default, for reference: its error is far
    below the cubic's and the bf16 rounding of P."""
    x = grid()
    rel = np.abs(run(x, 1) - np.exp2(x.astype(np.float64))) / np.exp2(x.astype(np.float64))
    assert rel.max() <= 2e-6, float(rel.max())


def test_cubic_below_the_normal_range_and_clamp():
    x = np.array([-126.5, -127.0, -127.5, -130.0, -1e4, -np.inf], np.float32)
    y = run(x, 0)
    assert np.all(np.isfinite(y)) and np.all(y >= 0.0) and np.all(y <= 2.0 ** -126)
