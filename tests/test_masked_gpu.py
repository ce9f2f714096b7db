"""Masked attention on the GPU (causal / sliding window, Nq != Nk, packed
batches) against the float64 masked oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import _lib, ops
from tests.parity import assert_grad, assert_lse, assert_o

pytestmark = pytest.mark.gpu

# (Nq, Nk, window_left, window_right): chunked prefill, more queries than keys
# (rows with no key), causal sliding windows, a two-sided local window, a left
# bound only, the diagonal alone, and a causal mask shifted right.
CASES = [
    (300, 1000, -1, 0),
    (1000, 300, -1, 0),
    (777, 777, 100, 0),
    (640, 640, 63, 0),
    (777, 777, 64, 64),
    (513, 2000, 200, -1),
    (1000, 1000, 0, 0),
    (384, 384, -1, 5),
    (1, 700, -1, 0),
    (129, 129, 1000, 0),
]


def _run(x, d, wl, wr, grads=True):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ops.fwd_masked(q, k, v, window=(wl, wr))
    out = {"o": o, "lse": lse}
    if grads:
        out["dq"], out["dk"], out["dv"] = ops.bwd_masked(q, k, v, o, lse, x["do"].cuda(), window=(wl, wr))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES)
def test_masked_forward_backward(d, case):
    Nq, Nk, wl, wr = case
    x = synth.make_masked(2, Nq, Nk, 4, 2, d, seed=Nq + Nk + wl)
    r = _run(x, d, wl, wr)
    f64 = {n: synth.to_f64(x[n]) for n in x}
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.masked_forward(f64["q"], f64["k"], f64["v"], scale, wl, wr)
    tag = f"Nq{Nq} Nk{Nk} w({wl},{wr}) d{d}"
    assert_o(synth.to_f64(r["o"]), o_ref, f"O {tag}")
    assert_lse(r["lse"].cpu().numpy(), l_ref, f"lse {tag}")
    refs = oracle.masked_backward(f64["q"], f64["k"], f64["v"], f64["do"], scale, wl, wr)
    for name, ref in zip(("dq", "dk", "dv"), refs):
        assert_grad(synth.to_f64(r[name]), ref, f"{name} {tag}")


@pytest.mark.parametrize("poly", [0, 4, 8, 16])
@pytest.mark.parametrize("d", [64, 128])
def test_window_forward_cubic_share(d, poly):
    """The sliding-window kernels at each share of exponentials on the cubic
    (one column pair in 8 or 16, or none; 1/4 runs as 1/8)."""
    x = synth.make_masked(2, 777, 777, 4, 2, d, seed=31 + d + poly)
    ops.set_option(_lib.FA_OPT_POLY_EXP, poly)
    try:
        r = _run(x, d, 100, 0, grads=False)
    finally:
        ops.set_option(_lib.FA_OPT_POLY_EXP, _lib.FA_POLY_EXP_DEFAULT)
    f64 = {n: synth.to_f64(x[n]) for n in x}
    o_ref, l_ref = oracle.masked_forward(f64["q"], f64["k"], f64["v"], 1.0 / math.sqrt(d), 100, 0)
    assert_o(synth.to_f64(r["o"]), o_ref, f"O window d{d} cubic 1/{poly}")
    assert_lse(r["lse"].cpu().numpy(), l_ref, f"lse window d{d} cubic 1/{poly}")


def test_rows_without_keys_and_unseen_keys():
    """Nq > Nk causal: the first Nq - Nk rows give O = 0, lse = -inf, dQ = 0;
    a narrow window leaves early keys unseen: dK = dV = 0 there."""
    x = synth.make_masked(1, 600, 200, 2, 2, 128, seed=9)
    r = _run(x, 128, -1, 0)
    assert torch.all(r["o"][:, :400] == 0) and torch.all(torch.isneginf(r["lse"][:, :, :400]))
    assert torch.all(r["dq"][:, :400] == 0)
    y = synth.make_masked(1, 128, 1000, 2, 1, 64, seed=10)
    s = _run(y, 64, 50, 0)
    first_seen = 1000 - 128 - 50
    assert torch.all(s["dk"][:, :first_seen] == 0) and torch.all(s["dv"][:, :first_seen] == 0)
    assert torch.any(s["dv"][:, first_seen:] != 0)


def test_no_keys_at_all():
    q = torch.randn(2, 70, 4, 128, device="cuda").to(torch.bfloat16)
    kv = torch.empty(2, 0, 4, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = ops.fwd_masked(q, kv, kv, causal=True)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("d", [64, 128])
def test_square_causal_is_bitwise_the_causal_call(d):
    x = synth.make_dense(2, 4, 700, d, seed=3)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o1, l1 = ops.fwd(q, k, v, causal=True)
    o2, l2 = ops.fwd_masked(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = ops.bwd(q, k, v, o1, l1, do, causal=True)
    g2 = ops.bwd_masked(q, k, v, o1, l1, do, causal=True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_window_past_the_sequence_is_no_window():
    x = synth.make_masked(1, 300, 500, 4, 4, 128, seed=4)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = ops.fwd_masked(q, k, v, window=(5000, 0))
    o2, l2 = ops.fwd_masked(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [(-1, 0), (96, 0), (-1, -1)])
def test_masked_varlen(d, window):
    """Chunked prefill on a packed batch: new queries of every sequence against
    its whole cache (lengths 1..900), one sequence with no query."""
    lq, lk = [1, 100, 300, 17, 0, 250], [50, 100, 900, 400, 30, 250]
    x = synth.make_masked_varlen(lq, lk, 4, 2, d, seed=sum(lq) + d)
    dev = {n: x[n].cuda() for n in x}
    wl, wr = window
    o, lse = ops.fwd_masked_varlen(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                                   max(lq), max(lk), window=window)
    dq, dk, dv = ops.bwd_masked_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], dev["cu_seqlens_q"],
                                       dev["cu_seqlens_k"], max(lq), max(lk), window=window)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    f64 = {n: synth.to_f64(x[n]) for n in ("q", "k", "v", "do")}
    cu_q, cu_k = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.masked_varlen_forward(f64["q"], f64["k"], f64["v"], cu_q, cu_k, scale, wl, wr)
    assert_o(synth.to_f64(o), o_ref, f"varlen O {window}")
    assert_lse(lse.cpu().numpy(), l_ref, f"varlen lse {window}")
    refs = oracle.masked_varlen_backward(f64["q"], f64["k"], f64["v"], f64["do"], cu_q, cu_k, scale, wl, wr)
    for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert_grad(synth.to_f64(g), ref, f"varlen {name} {window}")


def test_bad_packed_offsets_are_reported():
    """A key offset past the end of K is reported and that sequence is skipped."""
    lq, lk = [10, 20], [40, 30]
    x = synth.make_masked_varlen(lq, lk, 2, 2, 128, seed=2)
    dev = {n: x[n].cuda() for n in x}
    bad_k = dev["cu_seqlens_k"].clone()
    bad_k[2] = 1000  # total_k is 70
    ops.fwd_masked_varlen(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], bad_k, 20, 1000, causal=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0x2001
    assert ops.device_error() == 0


def test_sliding_window_long_sampled_rows():
    """8192 tokens, a causal window of 1024 (d = 128, 8 heads): sampled rows
    against the oracle over each row's own window of keys."""
    B, N, H, d, w = 1, 8192, 8, 128, 1023
    x = synth.make_dense(B, H, N, d, seed=11, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ops.fwd_masked(q, k, v, window=(w, 0))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    scale = 1.0 / math.sqrt(d)
    rows = [0, 1, 127, 128, 1023, 1024, 1025, 4000, 8191]
    for h in (0, 5):
        qh, kh, vh = (synth.to_f64(x[n][0, :, h]) for n in ("q", "k", "v"))
        vis = oracle.window_visible(N, N, w, 0)[rows]
        o_ref, l_ref = oracle.head_forward_visible(qh[rows], kh, vh, scale, vis)
        assert_o(synth.to_f64(o[0, rows, h]), o_ref, f"window rows h{h}")
        assert_lse(lse[0, h, rows].cpu().numpy(), l_ref, f"window rows h{h}")
