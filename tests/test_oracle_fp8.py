"""Pins of the FP8 oracle: the e4m3 format, the fast Walsh-Hadamard transform,
block quantisation, and the page's outlier ablation.

Facts pinned come from outside the oracle: the format's definition (largest
value 448, 3 mantissa bits), PyTorch's float8_e4m3fn conversion, SciPy's
Hadamard matrix, the identity H H^T = d I, the page's claim that a block
scale confines an outlier to its block, and the RMSE figures the page quotes.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import attention as A
from oracle import fp8 as F

RNG = np.random.default_rng(99)


# ------------------------------------------------------------------ e4m3

KNOWN = [  # value, code: from the format (sign | 4-bit exponent, bias 7 | 3-bit mantissa)
    (1.0, 0x38), (-2.0, 0xC0), (448.0, 0x7E), (-448.0, 0xFE), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01),
    (0.0, 0x00), (240.0, 0x77), (1.125, 0x39), (7 * 2.0 ** -9, 0x07), (0.875 * 2.0 ** -6, 0x07),
]


def check_known(encode):
    return all(int(encode(np.float32(v))) == c for v, c in KNOWN)


def check_saturation(encode):
    return int(encode(np.float32(1e6))) == 0x7E and int(encode(np.float32(-500.0))) == 0xFE \
        and int(encode(np.float32(464.0))) == 0x7E


def check_ties_to_even(encode):
    """The midpoint of two adjacent finite codes rounds to the one with an even mantissa."""
    vals = F.e4m3_decode(np.arange(0x7E + 1))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    got = encode(mids).astype(np.int64)
    want = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F))
    return bool(np.all(got == want))


def check_torch(encode):
    x = np.concatenate([RNG.standard_normal(50000) * 60, RNG.standard_normal(50000) * 0.01]).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return bool(np.all(encode(x) == ref))


def test_e4m3_known_codes():
    assert check_known(F.e4m3_encode)


def test_e4m3_saturates():
    assert check_saturation(F.e4m3_encode)


def test_e4m3_ties_to_even():
    assert check_ties_to_even(F.e4m3_encode)


def test_e4m3_matches_torch_in_range():
    assert check_torch(F.e4m3_encode)


def test_e4m3_round_trip_and_order():
    codes = np.arange(256)
    vals = F.e4m3_decode(codes)
    fin = np.isfinite(vals)
    assert fin.sum() == 254  # 0x7F and 0xFF are NaN
    back = F.e4m3_encode(vals[fin].astype(np.float32))
    assert np.all(back == codes[fin])
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0) and pos[-1] == 448.0


def mutant_encode_half_away(y):
    """Ties rounded away from zero instead of to even."""
    y = np.asarray(y, np.float32)
    out = F.e4m3_encode(y).astype(np.int64)
    vals = F.e4m3_decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2
    a = np.abs(y.astype(np.float64))
    mag = out & 0x7F
    down = np.isin(a, mids) & (F.e4m3_decode(mag) < a)
    return np.where(down, out + 1, out).astype(np.uint8)


def mutant_encode_no_saturation(y):
    y = np.asarray(y, np.float32)
    out = F.e4m3_encode(y)
    return np.where(np.abs(y) > 448, np.uint8(0x7F) | (np.signbit(y) << 7).astype(np.uint8), out).astype(np.uint8)


def mutant_encode_truncate(y):
    """Round toward zero."""
    y = np.asarray(y, np.float32)
    out = F.e4m3_encode(y)
    back = F.e4m3_decode(out)
    over = np.abs(back) > np.abs(y)
    return np.where(over, out - 1, out).astype(np.uint8)


@pytest.mark.parametrize("mutant", [mutant_encode_half_away, mutant_encode_no_saturation, mutant_encode_truncate])
def test_encode_mutants_are_rejected(mutant):
    assert not all([check_known(mutant), check_saturation(mutant), check_ties_to_even(mutant), check_torch(mutant)])


# ------------------------------------------------------------------ Walsh-Hadamard

@pytest.mark.parametrize("d", [64, 128])
def test_fwht_is_the_hadamard_product(d):
    x = RNG.standard_normal((5, d))
    assert np.allclose(F.fwht(x), x @ scipy.linalg.hadamard(d), atol=1e-12, rtol=0)


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_keeps_scores_up_to_d(d):
    """(x H D)(y H D)^T = d x y^T, since H H^T = d I and D D = I."""
    signs = np.where(RNG.random(d) < 0.5, -1.0, 1.0)
    x, y = RNG.standard_normal((7, d)), RNG.standard_normal((9, d))
    xr, yr = F.fwht(x) * signs, F.fwht(y) * signs
    assert np.allclose(xr @ yr.T, d * (x @ y.T), atol=1e-10, rtol=0)
    # hence attention over rotated operands with the scale divided by d is unchanged
    v = RNG.standard_normal((9, d))
    o1, l1 = A.head_forward(x, y, v, 0.3, False)
    o2, l2 = A.head_forward(xr, yr, v, 0.3 / d, False)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def test_fwht_f32_is_the_float64_transform_rounded():
    x = RNG.standard_normal((64, 128)).astype(np.float32)
    exact = F.fwht(x.astype(np.float64))
    got = F.fwht_f32(x).astype(np.float64)
    bound = 7 * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True) * 2
    assert np.all(np.abs(got - exact) <= bound)


def test_rotation_spreads_an_outlier():
    """A lone large coordinate is spread over all d coordinates: every entry of
    x H has the outlier's magnitude, so the row's peak-to-rms ratio drops from
    sqrt(d) to 1."""
    d = 128
    x = np.zeros(d, np.float32)
    x[17] = 50.0
    r = F.rotate_f32(x[None], np.ones(d))[0]
    assert np.all(np.abs(r) == 50.0)


# ------------------------------------------------------------------ block quantisation

def check_block_scales(quantize):
    """Scale = amax / 448, so the block's largest entry maps to code +-448."""
    x = RNG.standard_normal((1, 300, 2, 128)).astype(np.float32)
    codes, scales = quantize(x)
    ok = scales.shape == (1, 2, 3)
    for h in range(2):
        for t in range(3):
            blk = codes[0, 128 * t:128 * (t + 1), h]
            ok &= int((blk & 0x7F).max()) == 0x7E
            ok &= scales[0, h, t] == np.float32(np.abs(x[0, 128 * t:128 * (t + 1), h]).max() / np.float32(448))
    return bool(ok)


def check_outlier_stays_in_block(quantize):
    """An outlier in block 0 leaves block 1's scale untouched (the page's reason
    for block scales)."""
    x = RNG.standard_normal((1, 256, 1, 128)).astype(np.float32)
    _, s0 = quantize(x)
    y = x.copy()
    y[0, 5, 0, 3] = 1000.0
    _, s1 = quantize(y)
    return bool(s1[0, 0, 1] == s0[0, 0, 1] and s1[0, 0, 0] > 10 * s0[0, 0, 0])


def check_dequant_error(quantize):
    x = (RNG.standard_normal((1, 256, 1, 128)) * 3).astype(np.float32)
    codes, scales = quantize(x)
    xh = F.dequantize(codes, scales)
    sc = np.repeat(scales[0, 0], 128)[:, None]
    bound = np.maximum(2.0 ** -4 * np.abs(x[0, :, 0]), 2.0 ** -10 * sc)
    return bool(np.all(np.abs(xh[0, :, 0] - x[0, :, 0]) <= bound + 1e-12))


def test_block_scales():
    assert check_block_scales(F.fp8_quantize)


def test_outlier_stays_in_block():
    assert check_outlier_stays_in_block(F.fp8_quantize)


def test_dequantisation_error_bound():
    assert check_dequant_error(F.fp8_quantize)


def test_zero_block():
    codes, scales = F.fp8_quantize(np.zeros((1, 130, 1, 64), np.float32))
    assert np.all(codes == 0) and np.all(scales == 0.0)
    assert np.all(F.dequantize(codes, scales) == 0.0)


def mutant_quant_per_tensor(x, signs=None, block_rows=128):
    x = np.asarray(x, np.float32)
    amax = np.float32(np.abs(x).max())
    sc = np.float32(amax / np.float32(448))
    B, N, H, d = x.shape
    nblk = -(-N // block_rows)
    return F.e4m3_encode((x / sc).astype(np.float32)), np.full((B, H, nblk), sc, np.float32)


def mutant_quant_wrong_max(x, signs=None, block_rows=128):
    x = np.asarray(x, np.float32)
    B, N, H, d = x.shape
    nblk = -(-N // block_rows)
    codes = np.zeros(x.shape, np.uint8)
    scales = np.zeros((B, H, nblk), np.float32)
    for b in range(B):
        for h in range(H):
            for t in range(nblk):
                blk = x[b, 128 * t:128 * (t + 1), h]
                sc = np.float32(np.abs(blk).max() / np.float32(240))  # e4m3's max misremembered
                scales[b, h, t] = sc
                codes[b, 128 * t:128 * (t + 1), h] = F.e4m3_encode((blk / sc).astype(np.float32))
    return codes, scales


@pytest.mark.parametrize("mutant", [mutant_quant_per_tensor, mutant_quant_wrong_max])
def test_quantizer_mutants_are_rejected(mutant):
    assert not all([check_block_scales(mutant), check_outlier_stays_in_block(mutant)])


# ------------------------------------------------------------------ the page's outlier ablation

def _outlier_inputs(seed, B=1, N=1024, H=2, d=128):
    rng = np.random.default_rng(seed)

    def mk():
        a = rng.standard_normal((B, N, H, d))
        a = a + (rng.random((B, N, H, d)) < 0.001) * rng.standard_normal((B, N, H, d)) * 10.0  # N(0, 100)
        return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy()

    q, k, v = mk(), mk(), mk()
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    return q, k, v, signs


def test_outlier_ablation_matches_the_page():
    """Page: 9.1e-3 with block quantisation and incoherent processing,
    9.3e-3 without block quantisation, 2.4e-2 without incoherent processing
    and for per-tensor scaling.  Pinned: the full method's RMSE within 30% of
    9.1e-3; the rotation with per-tensor scales within 10% of the full method
    (block scales add little); the rotation cutting the error by at least 1.3x;
    per-tensor scales no better than block scales without the rotation.  The
    page's unrotated figure (2.4e-2) is not reproduced in size: these inputs
    give about 1.3e-2 (its sequence length and head size are not stated)."""
    for seed in (7, 8):
        q, k, v, signs = _outlier_inputs(seed)
        d = q.shape[-1]
        o_ref = A.forward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), d ** -0.5, False)[0]
        rmse = {}
        for name, s, blk in (("full", signs, True), ("tensor", None, False), ("block_no_rot", None, True),
                             ("tensor_rot", signs, False)):
            o = F.fp8_forward_variant(q, k, v, d ** -0.5, False, s, blk)
            rmse[name] = float(np.sqrt(np.mean((o - o_ref) ** 2)))
        assert 0.7 * 9.1e-3 <= rmse["full"] <= 1.3 * 9.1e-3, rmse
        assert abs(rmse["tensor_rot"] - rmse["full"]) <= 0.1 * rmse["full"], rmse
        assert rmse["block_no_rot"] >= 1.3 * rmse["full"], rmse
        assert rmse["tensor"] >= rmse["block_no_rot"], rmse


def test_fp8_forward_close_to_exact_without_outliers():
    q, k, v = (RNG.standard_normal((1, 300, 2, 128)).astype(np.float32) for _ in range(3))
    signs = np.where(RNG.random(128) < 0.5, -1.0, 1.0)
    o8, l8 = F.fp8_forward(q, k, v, 128 ** -0.5, True, signs)
    o, l = A.forward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), 128 ** -0.5, True)
    assert np.sqrt(np.mean((o8 - o) ** 2)) < 2e-2 and np.max(np.abs(l8 - l)) < 0.1


# ------------------------------------------------------------------ reciprocal scale vs the plain quotient

def quotient_codes(x32, signs=None, block_rows=128):
    """e4m3(x / scale) with the quotient rounded once to float32: the plain
    form of "divide by the block's scale" that the page's description implies
    before any choice of how a kernel evaluates it."""
    codes, scales = F.fp8_quantize(x32, signs, block_rows)
    B, N, H, d = x32.shape
    out = np.zeros_like(codes)
    for b in range(B):
        for h in range(H):
            rows = np.asarray(x32[b, :, h], np.float32)
            if signs is not None:
                rows = F.rotate_f32(rows, signs)
            for t, sc in enumerate(scales[b, h]):
                if sc == 0:
                    continue
                blk = rows[t * block_rows:(t + 1) * block_rows]
                out[b, t * block_rows:(t + 1) * block_rows, h] = F.e4m3_encode((blk / sc).astype(np.float32))
    return out, codes


def code_steps(a, b):
    """Distance between two e4m3 codes along the number line (codes of one
    sign are ordered by their low 7 bits); signs must agree unless both are 0."""
    a = a.astype(np.int64)
    b = b.astype(np.int64)
    va = np.where(a & 0x80, -(a & 0x7F), a & 0x7F)
    vb = np.where(b & 0x80, -(b & 0x7F), b & 0x7F)
    return np.abs(va - vb)


@pytest.mark.parametrize("rotate", [False, True])
def test_reciprocal_codes_within_one_step_of_the_quotient(rotate):
    """The quantiser multiplies by the float32 reciprocal of the scale
    (reading in the oracle's header).  Against the plain quotient x / scale
    the two float32 values differ by at most a couple of float32 ulps, so a
    code can move only where an e4m3 rounding midpoint lies between them: at
    most one code step, and only where the quotient sits on (or within a few
    float32 ulps of) a midpoint.  Unrotated bf16 inputs hit exact ties when
    the block maximum makes the scale a short binary fraction (24.5 / 448 =
    0.0546875, say): measured 7e-4 of elements here; the rotated (float32
    transform) inputs almost never do."""
    x = np.asarray(_outlier_inputs(11, B=2, N=2048, H=2, d=128)[0], np.float32)
    signs = np.where(np.random.default_rng(5).random(128) < 0.5, -1.0, 1.0).astype(np.float32) if rotate else None
    plain, recip = quotient_codes(x, signs)
    steps = code_steps(plain, recip)
    assert steps.max() <= 1
    frac = float(np.mean(steps > 0))
    assert frac <= (2e-3 if not rotate else 1e-4), frac
    # every differing element: the plain quotient lies within 4 float32 ulps of
    # the midpoint between the two codes' values
    codes, scales = F.fp8_quantize(x, signs)
    for b, n, h, c in np.argwhere(steps > 0):
        row = x[b, :, h] if signs is None else F.rotate_f32(x[b, :, h], signs)
        y = np.float32(row[n, c] / scales[b, h, n // 128])
        mid = 0.5 * (F.e4m3_decode(plain[b, n, h, c]) + F.e4m3_decode(recip[b, n, h, c]))
        assert abs(float(y) - mid) <= 4 * float(np.spacing(np.abs(y))), (float(y), mid)
