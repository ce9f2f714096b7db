"""Guard bands around every output buffer: the stand-in for a memory checker
on this GPU pool.  Each output (O, lse, dQ, dK, dV, the decode outputs and the
workspaces) is a view into a larger device buffer whose bytes are all set to
a sentinel first; after the call every byte outside the view must still be
the sentinel, and the view must hold exactly what the ordinary call (with
plainly allocated outputs) produces.  The cases are the ones whose writes are
guarded by row and sequence bounds: ragged lengths, packed batches with empty
sequences, rows that see no key, keys that no query sees, paged caches with
partly filled last pages.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from exact_attention_94_gb300 import _lib, ops

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5
GUARD = 4096  # bytes before and after each view (a multiple of 16: views stay 16-byte aligned)


class Guarded:
    """A tensor of `shape` and `dtype` carved out of a sentinel-filled buffer,
    `shift` bytes past the guard band (a multiple of 16)."""

    def __init__(self, shape, dtype, shift=0):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.nbytes = n
        self.lo = GUARD + shift
        self.buf = torch.full((self.lo + n + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.buf[self.lo:self.lo + n].view(dtype).view(shape) if n else torch.empty(shape, dtype=dtype,
                                                                                              device="cuda")

    def check(self, what):
        torch.cuda.synchronize()
        head = self.buf[:self.lo]
        tail = self.buf[self.lo + self.nbytes:]
        bad_h = int((head != SENTINEL).sum())
        bad_t = int((tail != SENTINEL).sum())
        assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} bytes before and {bad_t} after the buffer changed"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _same(a, b, what):
    assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                       b.view(torch.uint8) if b.dtype != torch.uint8 else b), f"{what}: differs from the plain call"


def _bitwise_or_both_nan(a, b, what):
    """Equal bits; lse may hold -inf, which compares fine bit for bit."""
    _same(a.contiguous(), b.contiguous(), what)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 257])
def test_dense_forward_backward_stay_in_bounds(d, causal, N):
    B, H = 2, 3
    x = synth.make_dense(B, H, N, d, seed=N + d, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o_ref, l_ref = ops.fwd(q, k, v, causal=causal)
    o, lse = Guarded(q.shape, torch.bfloat16), Guarded((B, H, N), torch.float32)
    ops.fwd(q, k, v, causal=causal, out=o.t, lse=lse.t)
    o.check("O")
    lse.check("lse")
    _same(o.t, o_ref, "O")
    _bitwise_or_both_nan(lse.t, l_ref, "lse")
    # the backward's dQ is accumulated with atomics (order not fixed): compare within rounding
    ref = ops.bwd(q, k, v, o_ref, l_ref, do, causal=causal)
    g = [Guarded(q.shape, torch.bfloat16) for _ in range(3)]
    ws = Guarded((ops.lib().fa_bwd_workspace_bytes(B, H, N, d),), torch.uint8)
    ops.bwd(q, k, v, o_ref, l_ref, do, causal=causal, workspace=ws.t, out=tuple(x.t for x in g))
    for name, gg, r in zip(("dq", "dk", "dv"), g, ref):
        gg.check(name)
        assert torch.allclose(gg.t.float(), r.float(), rtol=2e-2, atol=1e-3), name
    ws.check("workspace")
    assert ops.device_error() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_outputs_16_but_not_32_byte_aligned(d):
    """Rows of O, dK and dV are written 32 bytes per store when their address
    allows it and 16 bytes per store otherwise: outputs placed 16 bytes off a
    32-byte boundary take the second path, with the same results and nothing
    written outside."""
    B, H, N = 2, 3, 257
    x = synth.make_dense(B, H, N, d, seed=77, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o_ref, l_ref = ops.fwd(q, k, v, causal=True)
    o, lse = Guarded(q.shape, torch.bfloat16, shift=16), Guarded((B, H, N), torch.float32, shift=16)
    assert o.t.data_ptr() % 32 == 16
    ops.fwd(q, k, v, causal=True, out=o.t, lse=lse.t)
    o.check("O")
    lse.check("lse")
    _same(o.t, o_ref, "O")
    _bitwise_or_both_nan(lse.t, l_ref, "lse")
    ref = ops.bwd(q, k, v, o_ref, l_ref, do, causal=True)
    g = [Guarded(q.shape, torch.bfloat16, shift=16) for _ in range(3)]
    ops.bwd(q, k, v, o_ref, l_ref, do, causal=True, out=tuple(t.t for t in g))
    for name, gg, r in zip(("dq", "dk", "dv"), g, ref):
        gg.check(name)
        if name == "dq":
            assert torch.allclose(gg.t.float(), r.float(), rtol=2e-2, atol=1e-3), name
        else:
            _same(gg.t, r, name)
    assert ops.device_error() == 0


def test_varlen_with_empty_sequences_stays_in_bounds():
    lengths = [200, 0, 64, 0, 385, 1]
    H, d = 2, 128
    x = synth.make_varlen(lengths, H, d, seed=3, device="cuda")
    cu = x["cu_seqlens"].cuda()
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    total, mx = sum(lengths), max(lengths)
    o_ref, l_ref = ops.fwd_varlen(q, k, v, cu, mx, causal=True)
    o, lse = Guarded(q.shape, torch.bfloat16), Guarded((H, total), torch.float32)
    st = ops.lib().fa_fwd_varlen(_p(q), _p(k), _p(v), _p(o.t), _p(lse.t), _p(cu), len(lengths), mx, total, H, d, 1,
                                 1.0 / math.sqrt(d), _s())
    assert st == _lib.FA_OK
    o.check("varlen O")
    lse.check("varlen lse")
    _same(o.t, o_ref, "varlen O")
    _bitwise_or_both_nan(lse.t, l_ref, "varlen lse")
    g = [Guarded(q.shape, torch.bfloat16) for _ in range(3)]
    ws = Guarded((ops.lib().fa_bwd_varlen_workspace_bytes(total, H, d),), torch.uint8)
    st = ops.lib().fa_bwd_varlen(_p(q), _p(k), _p(v), _p(o_ref), _p(l_ref), _p(do), _p(g[0].t), _p(g[1].t),
                                 _p(g[2].t), _p(ws.t), _p(cu), len(lengths), mx, total, H, d, 1, 1.0 / math.sqrt(d),
                                 _s())
    assert st == _lib.FA_OK
    ref = ops.bwd_varlen(q, k, v, o_ref, l_ref, do, cu, mx, causal=True)
    for name, gg, r in zip(("dq", "dk", "dv"), g, ref):
        gg.check(f"varlen {name}")
        assert torch.allclose(gg.t.float(), r.float(), rtol=2e-2, atol=1e-3), name
    ws.check("varlen workspace")
    assert ops.device_error() == 0


@pytest.mark.parametrize("window", [(-1, 0), (16, 0), (3, 5)])
def test_rows_without_keys_stay_in_bounds(window):
    """Nq > Nk with a bottom-right causal mask: the first Nq - Nk rows see no
    key (O = 0, lse = -inf); with windows, keys that no query sees get dK = dV = 0."""
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 2, 300, 130, 64
    x = synth.make_masked(B, Nq, Nk, Hq, Hkv, d, seed=8, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    wl, wr = window
    o_ref, l_ref = ops.fwd_masked(q, k, v, window=window)
    o, lse = Guarded(q.shape, torch.bfloat16), Guarded((B, Hq, Nq), torch.float32)
    st = ops.lib().fa_fwd_masked(_p(q), _p(k), _p(v), _p(o.t), _p(lse.t), B, Hq, Hkv, Nq, Nk, d, wl, wr,
                                 1.0 / math.sqrt(d), _s())
    assert st == _lib.FA_OK
    o.check("masked O")
    lse.check("masked lse")
    _same(o.t, o_ref, "masked O")
    _bitwise_or_both_nan(lse.t, l_ref, "masked lse")
    ref = ops.bwd_masked(q, k, v, o_ref, l_ref, do, window=window)
    gq = Guarded(q.shape, torch.bfloat16)
    gk, gv = Guarded(k.shape, torch.bfloat16), Guarded(v.shape, torch.bfloat16)
    ws = Guarded((ops.lib().fa_bwd_workspace_bytes(B, Hq, Nq, d),), torch.uint8)
    st = ops.lib().fa_bwd_masked(_p(q), _p(k), _p(v), _p(o_ref), _p(l_ref), _p(do), _p(gq.t), _p(gk.t), _p(gv.t),
                                 _p(ws.t), B, Hq, Hkv, Nq, Nk, d, wl, wr, 1.0 / math.sqrt(d), _s())
    assert st == _lib.FA_OK
    for name, gg, r in zip(("dq", "dk", "dv"), (gq, gk, gv), ref):
        gg.check(f"masked {name}")
        assert torch.allclose(gg.t.float(), r.float(), rtol=2e-2, atol=1e-3), name
    ws.check("masked workspace")
    assert ops.device_error() == 0


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_and_paged_decode_stay_in_bounds(splits):
    B, H, L, d = 3, 4, 333, 128
    x = synth.make_decode(B, H, L, d, seed=9, device="cuda")
    q, k, v = x["q"], x["k"], x["v"]
    o_ref, l_ref = ops.decode(q, k, v, num_splits=splits)
    o, lse = Guarded(q.shape, torch.bfloat16), Guarded((B, H), torch.float32)
    ws = Guarded((ops.lib().fa_decode_workspace_bytes(B, H, d, splits),), torch.uint8)
    st = ops.lib().fa_decode_splitkv(_p(q), _p(k), _p(v), _p(o.t), _p(lse.t), B, H, L, d, splits, _p(ws.t),
                                     1.0 / math.sqrt(d), _s())
    assert st == _lib.FA_OK
    for g, name in ((o, "decode O"), (lse, "decode lse"), (ws, "decode workspace")):
        g.check(name)
    _same(o.t, o_ref, "decode O")
    _same(lse.t, l_ref, "decode lse")
    # paged: ragged lengths, the last page of most sequences partly filled
    lengths = [1, 15, 17, 100]
    xp = synth.make_paged_decode(lengths, H, d, page_size=16, seed=10, device="cuda")
    bt, sl = xp["block_table"].cuda(), xp["seq_lens"].cuda()
    Bp = len(lengths)
    op_ref, lp_ref = ops.decode_paged(xp["q"], xp["k_pages"], xp["v_pages"], bt, sl, max(lengths),
                                      num_splits=splits)
    op, lp = Guarded((Bp, 1, H, d), torch.bfloat16), Guarded((Bp, H), torch.float32)
    wsp = Guarded((ops.lib().fa_decode_workspace_bytes(Bp, H, d, splits),), torch.uint8)
    st = ops.lib().fa_decode_paged(_p(xp["q"]), _p(xp["k_pages"]), _p(xp["v_pages"]), _p(bt), _p(sl), _p(op.t),
                                   _p(lp.t), Bp, H, d, 16, xp["k_pages"].shape[0], bt.shape[1], max(lengths), splits,
                                   _p(wsp.t), 1.0 / math.sqrt(d), _s())
    assert st == _lib.FA_OK
    for g, name in ((op, "paged O"), (lp, "paged lse"), (wsp, "paged workspace")):
        g.check(name)
    _same(op.t, op_ref, "paged O")
    _same(lp.t, lp_ref, "paged lse")
    assert ops.device_error() == 0
