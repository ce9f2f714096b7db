"""The bounds-checked test build (build.build_bounds(): the forward, backward
and decode kernels compiled with FA_BOUNDS_CHECK) on the cases whose accesses
are guarded by row, sequence and page bounds: ragged lengths, packed batches
with empty sequences, rows that see no key, keys that no query sees, e4m3
scales, split and paged decode with partly filled pages.

In that build every plain (non-TMA) global load, store and atomic of those
kernels checks its index against its buffer and, instead of touching memory
outside it, records code 0x3000 + site in the device error word.  Each case
runs through both libraries: the bounds-checked one must report no error and
produce what the product library produces (bit for bit, except dQ, which is
accumulated with atomics in no fixed order and is compared within rounding).
Together with the guard bands of test_canary_gpu.py this stands in for a
memory checker; the checks' own firing is not exercised, since no valid input
reaches them.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from exact_attention_94_gb300 import _lib, build

pytestmark = pytest.mark.gpu


def _load(path):
    lib = ctypes.CDLL(path)
    for name, (res, args) in _lib.SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


@pytest.fixture(scope="module")
def libs():
    return {"product": _lib.load(), "bounds": _load(build.build_bounds())}


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _device_error(lib):
    code = ctypes.c_uint(0)
    lib.fa_device_error(ctypes.byref(code))
    return code.value


def _both(libs, run):
    """run(lib) -> dict of output tensors, for each library; asserts the status
    and that the bounds-checked build recorded nothing."""
    out = {}
    for name, lib in libs.items():
        assert _device_error(lib) == 0
        res = run(lib)
        torch.cuda.synchronize()
        code = _device_error(lib)
        assert code == 0, f"{name}: device error {code:#x}"
        out[name] = res
    return out["product"], out["bounds"]


def _same(a, b, what):
    assert a.shape == b.shape and torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), \
        f"{what}: the bounds-checked build differs"


def _close(a, b, what):
    a, b = a.float(), b.float()
    err = float((a - b).norm() / max(float(b.norm()), 1e-6))
    assert err <= 1e-3, f"{what}: relative difference {err:.2e}"


def _compare(ref, got, atomics=("dq",)):
    for k in ref:
        (_close if k in atomics else _same)(got[k], ref[k], k)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 257])
def test_dense(libs, d, causal, N):
    B, H = 2, 3
    x = synth.make_dense(B, H, N, d, seed=N + d, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    sc = 1.0 / math.sqrt(d)

    def run(lib):
        o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        assert lib.fa_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, int(causal), sc, _s()) == _lib.FA_OK
        g = [torch.empty_like(q) for _ in range(3)]
        ws = torch.empty(lib.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
        assert lib.fa_bwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), *(_p(t) for t in g), _p(ws), B, H, N, d,
                          int(causal), sc, _s()) == _lib.FA_OK
        return dict(o=o, lse=lse, dq=g[0], dk=g[1], dv=g[2])

    _compare(*_both(libs, run))


@pytest.mark.parametrize("causal", [False, True])
def test_packed_with_empty_sequences(libs, causal):
    lengths = [200, 0, 64, 0, 385, 1, 700]
    H, d = 2, 128
    x = synth.make_varlen(lengths, H, d, seed=3, device="cuda")
    cu = x["cu_seqlens"].cuda()
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    total, mx, n = sum(lengths), max(lengths), len(lengths)
    sc = 1.0 / math.sqrt(d)

    def run(lib):
        o, lse = torch.empty_like(q), torch.empty((H, total), dtype=torch.float32, device="cuda")
        assert lib.fa_fwd_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu), n, mx, total, H, d, int(causal), sc,
                                 _s()) == _lib.FA_OK
        g = [torch.empty_like(q) for _ in range(3)]
        ws = torch.empty(lib.fa_bwd_varlen_workspace_bytes(total, H, d), dtype=torch.uint8, device="cuda")
        assert lib.fa_bwd_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), *(_p(t) for t in g), _p(ws), _p(cu), n,
                                 mx, total, H, d, int(causal), sc, _s()) == _lib.FA_OK
        return dict(o=o, lse=lse, dq=g[0], dk=g[1], dv=g[2])

    _compare(*_both(libs, run))


@pytest.mark.parametrize("window", [(-1, 0), (16, 0), (3, 5)])
def test_rows_without_keys_and_unseen_keys(libs, window):
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 2, 300, 130, 64
    x = synth.make_masked(B, Nq, Nk, Hq, Hkv, d, seed=8, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    wl, wr = window
    sc = 1.0 / math.sqrt(d)

    def run(lib):
        o, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
        assert lib.fa_fwd_masked(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Nq, Nk, d, wl, wr, sc,
                                 _s()) == _lib.FA_OK
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(lib.fa_bwd_workspace_bytes(B, Hq, Nq, d), dtype=torch.uint8, device="cuda")
        assert lib.fa_bwd_masked(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(gq), _p(gk), _p(gv), _p(ws), B, Hq,
                                 Hkv, Nq, Nk, d, wl, wr, sc, _s()) == _lib.FA_OK
        return dict(o=o, lse=lse, dq=gq, dk=gk, dv=gv)

    _compare(*_both(libs, run))


def test_packed_masked_chunked_prefill(libs):
    """Packed queries against longer packed caches (bottom-right causal, GQA)."""
    lq, lk = [1, 130, 0, 77], [5, 300, 64, 77]
    Hq, Hkv, d = 4, 2, 128
    g = torch.Generator().manual_seed(12)
    tq, tk = sum(lq), sum(lk)
    q = torch.randn((tq, Hq, d), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((tk, Hkv, d), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((tk, Hkv, d), generator=g).to(torch.bfloat16).cuda()
    do = torch.randn((tq, Hq, d), generator=g).to(torch.bfloat16).cuda()
    cq = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32).cuda()
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32).cuda()
    n, sc = len(lq), 1.0 / math.sqrt(d)

    def run(lib):
        o, lse = torch.empty_like(q), torch.empty((Hq, tq), dtype=torch.float32, device="cuda")
        assert lib.fa_fwd_masked_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cq), _p(ck), n, max(lq), max(lk), tq,
                                        tk, Hq, Hkv, d, -1, 0, sc, _s()) == _lib.FA_OK
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(lib.fa_bwd_varlen_workspace_bytes(tq, Hq, d), dtype=torch.uint8, device="cuda")
        assert lib.fa_bwd_masked_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(gq), _p(gk), _p(gv), _p(ws),
                                        _p(cq), _p(ck), n, max(lq), max(lk), tq, tk, Hq, Hkv, d, -1, 0, sc,
                                        _s()) == _lib.FA_OK
        return dict(o=o, lse=lse, dq=gq, dk=gk, dv=gv)

    _compare(*_both(libs, run))


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_and_paged_decode(libs, splits):
    B, H, L, d = 3, 4, 333, 128
    x = synth.make_decode(B, H, L, d, seed=9, device="cuda")
    q, k, v = x["q"], x["k"], x["v"]
    sc = 1.0 / math.sqrt(d)

    def run(lib):
        o, lse = torch.empty_like(q), torch.empty((B, H), dtype=torch.float32, device="cuda")
        ws = torch.empty(lib.fa_decode_workspace_bytes(B, H, d, splits), dtype=torch.uint8, device="cuda")
        assert lib.fa_decode_splitkv(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, L, d, splits, _p(ws), sc,
                                     _s()) == _lib.FA_OK
        return dict(o=o, lse=lse)

    _compare(*_both(libs, run))
    # paged: ragged lengths, the last page of most sequences partly filled
    lengths = [1, 15, 17, 100]
    xp = synth.make_paged_decode(lengths, H, d, page_size=16, seed=10, device="cuda")
    bt, sl = xp["block_table"].cuda(), xp["seq_lens"].cuda()
    Bp = len(lengths)

    def run_paged(lib):
        o, lse = torch.empty((Bp, 1, H, d), dtype=torch.bfloat16, device="cuda"), torch.empty(
            (Bp, H), dtype=torch.float32, device="cuda")
        ws = torch.empty(lib.fa_decode_workspace_bytes(Bp, H, d, splits), dtype=torch.uint8, device="cuda")
        assert lib.fa_decode_paged(_p(xp["q"]), _p(xp["k_pages"]), _p(xp["v_pages"]), _p(bt), _p(sl), _p(o), _p(lse),
                                   Bp, H, d, 16, xp["k_pages"].shape[0], bt.shape[1], max(lengths), splits, _p(ws), sc,
                                   _s()) == _lib.FA_OK
        return dict(o=o, lse=lse)

    _compare(*_both(libs, run_paged))


@pytest.mark.parametrize("window", [(-1, 0), (-1, -1), (100, 0)])
def test_fp8_forward(libs, window):
    """The e4m3 forward reads per-block scales of Q, K and V: a ragged
    length leaves a partly filled last block."""
    from exact_attention_94_gb300 import ops
    B, N, H, d = 1, 300, 2, 128
    x = synth.make_dense(B, H, N, d, seed=21, device="cuda", with_do=False)
    signs = synth.hadamard_signs(d, seed=1).cuda()
    qc, qs = ops.fp8_quantize(x["q"], signs)
    kc, ks = ops.fp8_quantize(x["k"], signs)
    vc, vs = ops.fp8_quantize(x["v"], None, transpose=True)
    wl, wr = window
    sc = 1.0 / math.sqrt(d)

    def run(lib):
        o, lse = torch.empty_like(x["q"]), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        assert lib.fa_fwd_fp8(_p(qc), _p(kc), _p(vc), _p(qs), _p(ks), _p(vs), _p(o), _p(lse), B, H, H, N, N, d, wl, wr,
                              1, sc, _s()) == _lib.FA_OK
        return dict(o=o, lse=lse)

    _compare(*_both(libs, run))
