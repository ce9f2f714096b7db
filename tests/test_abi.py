"""The C-ABI library: it builds, loads, exports every declared symbol, and its
host-side validation rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from exact_attention_94_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert "fa_fwd" in syms and "fa_decode_splitkv" in syms
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) <= set(_lib.SIGNATURES), set(syms) - set(_lib.SIGNATURES)


def test_status_strings(lib):
    assert _lib.status_string(0) == "FA_OK"
    assert _lib.status_string(5) == "FA_ERR_TIMEOUT"


P = ctypes.c_void_p
A = P(4096)          # fake, 16-byte aligned (never dereferenced: validation fails first)
MIS = P(4096 + 2)


def fwd(lib, q=A, d=128, N=16, B=1, H=1, causal=0, scale=0.1, o=A):
    return lib.fa_fwd(q, A, A, o, A, B, H, N, d, causal, scale, P(0))


def test_fwd_validation(lib):
    assert fwd(lib, d=96) == _lib.FA_ERR_UNSUPPORTED
    assert fwd(lib, d=256) == _lib.FA_ERR_UNSUPPORTED
    assert fwd(lib, q=P(0)) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, q=MIS) == _lib.FA_ERR_MISALIGNED
    assert fwd(lib, o=MIS) == _lib.FA_ERR_MISALIGNED
    assert fwd(lib, scale=0.0) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, causal=2) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, B=0) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, N=-1) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, N=0) == _lib.FA_OK            # empty input: nothing to do
    assert fwd(lib, N=65536 * 256) == _lib.FA_ERR_INVALID_ARG  # grid limit


def test_varlen_validation(lib):
    f = lib.fa_fwd_varlen
    assert f(A, A, A, A, A, P(0), 2, 8, 16, 1, 128, 0, 0.1, P(0)) == _lib.FA_ERR_INVALID_ARG
    assert f(A, A, A, A, A, A, 0, 8, 16, 1, 128, 0, 0.1, P(0)) == _lib.FA_ERR_INVALID_ARG
    assert f(A, A, A, A, A, A, 2, 8, 16, 1, 80, 0, 0.1, P(0)) == _lib.FA_ERR_UNSUPPORTED
    assert f(A, A, A, A, A, A, 2, 8, 0, 1, 128, 0, 0.1, P(0)) == _lib.FA_OK


def test_workspace_sizes(lib):
    B, H, N, d = 2, 3, 100, 64
    ws = lib.fa_bwd_workspace_bytes(B, H, N, d)
    assert ws >= B * H * N * d * 4 + B * H * N * 4
    assert lib.fa_bwd_varlen_workspace_bytes(N, H, d) >= N * H * d * 4 + H * N * 4
    assert lib.fa_decode_workspace_bytes(4, 8, 128, 3) >= 4 * 8 * 3 * (128 + 1) * 4
    assert lib.fa_decode_workspace_bytes(0, 8, 128, 3) == 0


def test_options(lib):
    assert lib.fa_set_option(_lib.FA_OPT_RESCALE_TAU, -1.0) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_set_option(_lib.FA_OPT_RESCALE_TAU, 8.0) == _lib.FA_OK
    assert lib.fa_set_option(99, 1.0) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_set_option(_lib.FA_OPT_WAIT_TIMEOUT_MS, 0.0) == _lib.FA_ERR_INVALID_ARG
    for share in (0.0, 1.0, 4.0, 8.0, 16.0):  # the cubic's share: none, default, one pair in 4 / 8 / 16
        assert lib.fa_set_option(_lib.FA_OPT_POLY_EXP, share) == _lib.FA_OK
    for share in (2.0, 3.0, -1.0, 32.0):
        assert lib.fa_set_option(_lib.FA_OPT_POLY_EXP, share) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_set_option(_lib.FA_OPT_POLY_EXP, _lib.FA_POLY_EXP_DEFAULT) == _lib.FA_OK  # back to the default


def test_masked_validation(lib):
    def f(wl=-1, wr=0, d=128, Nq=16, Nk=32, Hq=4, Hkv=2, q=A):
        return lib.fa_fwd_masked(q, A, A, A, A, 1, Hq, Hkv, Nq, Nk, d, wl, wr, 0.1, P(0))
    assert f(wl=-2) == _lib.FA_ERR_INVALID_ARG
    assert f(wr=-7) == _lib.FA_ERR_INVALID_ARG
    assert f(d=96) == _lib.FA_ERR_UNSUPPORTED
    assert f(Hkv=3) == _lib.FA_ERR_INVALID_ARG
    assert f(q=MIS) == _lib.FA_ERR_MISALIGNED
    assert f(Nq=0) == _lib.FA_OK
    b = lib.fa_bwd_masked
    assert b(A, A, A, A, A, A, A, A, A, A, 1, 4, 2, 16, 32, 128, -3, 0, 0.1, P(0)) == _lib.FA_ERR_INVALID_ARG
    assert b(A, A, A, A, A, A, A, A, A, A, 1, 4, 2, 0, 32, 128, -1, 0, 0.1, P(0)) == _lib.FA_ERR_INVALID_ARG
    fv = lib.fa_fwd_masked_varlen
    assert fv(A, A, A, A, A, P(0), A, 2, 8, 8, 16, 16, 2, 2, 128, -1, 0, 0.1, P(0)) == _lib.FA_ERR_INVALID_ARG
    assert fv(A, A, A, A, A, A, MIS, 2, 8, 8, 16, 16, 2, 2, 128, -1, 0, 0.1, P(0)) == _lib.FA_ERR_MISALIGNED
    assert fv(A, A, A, A, A, A, A, 2, 8, 0, 16, 16, 2, 2, 128, -1, 0, 0.1, P(0)) == _lib.FA_ERR_INVALID_ARG
    assert fv(A, A, A, A, A, A, A, 2, 8, 8, 0, 16, 2, 2, 128, -1, 0, 0.1, P(0)) == _lib.FA_OK
