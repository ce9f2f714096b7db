"""Forward parity: the CUDA path through the C ABI against the float64 oracle,
element by element, on seeded inputs shared by both sides."""
import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import _lib, ops
from tests.parity import assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_94_gb300 import build
    build.build()
    # the library's defaults: threshold 8, one column pair in 16 on the cubic
    ops.set_option(_lib.FA_OPT_RESCALE_TAU, 8.0)
    ops.set_option(_lib.FA_OPT_POLY_EXP, _lib.FA_POLY_EXP_DEFAULT)
    yield
    ops.set_option(_lib.FA_OPT_RESCALE_TAU, 8.0)
    ops.set_option(_lib.FA_OPT_POLY_EXP, _lib.FA_POLY_EXP_DEFAULT)


def run_dense(B, H, N, d, causal, seed=0, k_boost=1.0):
    x = synth.make_dense(B, H, N, d, seed=seed, k_boost=k_boost, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ops.fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    return x, synth.to_f64(o), lse.cpu().numpy()


def check_dense(B, H, N, d, causal, seed=0, k_boost=1.0):
    x, o, lse = run_dense(B, H, N, d, causal, seed, k_boost)
    o_ref, l_ref = oracle.forward(synth.to_f64(x["q"]), synth.to_f64(x["k"]), synth.to_f64(x["v"]),
                                  1.0 / np.sqrt(d), causal)
    assert_o(o, o_ref, f"O B{B} H{H} N{N} d{d} causal={causal}")
    assert_lse(lse, l_ref, f"lse B{B} H{H} N{N} d{d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload(causal):
    w = synth.WORKLOADS["tiny_causal" if causal else "tiny"]
    check_dense(w.B, w.H, w.N, w.d, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 257, 383, 640])
def test_ragged_lengths(d, causal, N):
    check_dense(1, 2, N, d, causal, seed=N)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_several_tiles_with_max_jumps(d, causal):
    # K x 3 in half of the heads: the running maximum jumps across tiles
    check_dense(2, 4, 1536 + 77, d, causal, seed=7, k_boost=3.0)


@pytest.mark.parametrize("tau", [0.0, 8.0, 30.0])
@pytest.mark.parametrize("poly", [0, 4, 8, 16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_threshold_and_exp_split(tau, poly, d, causal):
    """Every lazy-rescale threshold and every share of exponentials on the
    FMA-pipe cubic (0 = none, else one column pair in `poly`) gives the same
    result within tolerance, at both head dims, with and without the mask."""
    ops.set_option(_lib.FA_OPT_RESCALE_TAU, tau)
    ops.set_option(_lib.FA_OPT_POLY_EXP, poly)
    try:
        check_dense(1, 4, 1024 + 33, d, causal, seed=3, k_boost=3.0)
    finally:
        ops.set_option(_lib.FA_OPT_RESCALE_TAU, 8.0)
        ops.set_option(_lib.FA_OPT_POLY_EXP, _lib.FA_POLY_EXP_DEFAULT)


def test_large_score_offsets():
    """Scores around +-60 (scale 1): online softmax must subtract the maximum."""
    B, H, N, d = 1, 2, 512, 64
    x = synth.make_dense(B, H, N, d, seed=11, with_do=False)
    q = (x["q"].float() * 8).to(torch.bfloat16)
    o, lse = ops.fwd(q.cuda(), x["k"].cuda(), x["v"].cuda(), causal=False, scale=1.0)
    o_ref, l_ref = oracle.forward(synth.to_f64(q), synth.to_f64(x["k"]), synth.to_f64(x["v"]), 1.0, False)
    assert_o(synth.to_f64(o), o_ref, "large offsets O")
    assert_lse(lse.cpu().numpy(), l_ref, "large offsets lse")


def test_empty_is_noop():
    q = torch.empty((1, 0, 2, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = ops.fwd(q, q, q)
    assert o.numel() == 0 and lse.numel() == 0


def test_mid_workload_sampled_heads():
    """Full size (B16 H16 N2048 d64, non-causal), six (b, h) pairs compared in full."""
    w = synth.WORKLOADS["mid"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=w.seed, with_do=False, device="cuda")
    o, lse = ops.fwd(x["q"], x["k"], x["v"], causal=False)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (3, 15), (7, 8), (11, 2), (15, 15), (15, 0)]:
        qh, kh, vh = (synth.to_f64(x[n][b, :, h]) for n in ("q", "k", "v"))
        oh, lh = oracle.head_forward(qh, kh, vh, w.scale, False)
        assert_o(synth.to_f64(o[b, :, h]), oh, f"mid b{b} h{h}")
        assert_lse(lse[b, h].cpu().numpy(), lh, f"mid b{b} h{h}")


def test_long_workload_sampled_rows():
    """Full size (B2 H16 N8192 d128, causal, K x 3 in heads 0-7): four heads
    (two boosted), 384 sampled rows each, including the first and last rows."""
    w = synth.WORKLOADS["long"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=w.seed, k_boost=w.k_boost, with_do=False, device="cuda")
    o, lse = ops.fwd(x["q"], x["k"], x["v"], causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for b, h in [(0, 0), (1, 7), (0, 8), (1, 15)]:
        rows = np.unique(np.concatenate([[0, 1, 127, 128, 8191], rng.integers(0, w.N, 379)]))
        qh = synth.to_f64(x["q"][b, rows, h])
        kh, vh = synth.to_f64(x["k"][b, :, h]), synth.to_f64(x["v"][b, :, h])
        oh, lh = oracle.head_forward(qh, kh, vh, w.scale, True, q_pos=rows)
        assert_o(synth.to_f64(o[b, rows, h]), oh, f"long b{b} h{h}")
        assert_lse(lse[b, h, rows].cpu().numpy(), lh, f"long b{b} h{h}")
