"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI) against
the float64 oracle's gradients, relative Frobenius error <= 2e-2."""
import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import ops
from tests.parity import assert_grad

pytestmark = pytest.mark.gpu


def gpu_grads_dense(x, causal, device="cuda"):
    q, k, v, do = (x[n].to(device) for n in ("q", "k", "v", "do"))
    o, lse = ops.fwd(q, k, v, causal=causal)
    dq, dk, dv = ops.bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    return dq, dk, dv


def check_dense_bwd(B, H, N, d, causal, seed=0, k_boost=1.0):
    x = synth.make_dense(B, H, N, d, seed=seed, k_boost=k_boost)
    got = gpu_grads_dense(x, causal)
    ref = oracle.backward(*(synth.to_f64(x[n]) for n in ("q", "k", "v", "do")), 1.0 / np.sqrt(d), causal)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert_grad(synth.to_f64(g), r, f"{name} B{B} H{H} N{N} d{d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload(causal):
    w = synth.WORKLOADS["tiny_causal" if causal else "tiny"]
    check_dense_bwd(w.B, w.H, w.N, w.d, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 256, 300, 640])
def test_ragged_lengths(d, causal, N):
    check_dense_bwd(1, 2, N, d, causal, seed=100 + N)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_several_tiles_with_max_jumps(d, causal):
    check_dense_bwd(2, 3, 1024 + 45, d, causal, seed=17, k_boost=3.0)


def test_per_head_gradients_independent():
    """Two batch entries and heads never mix: the gradient of one head equals
    the single-head call on that head alone."""
    x = synth.make_dense(2, 3, 384, 128, seed=23)
    full = gpu_grads_dense(x, True)
    for b, h in [(0, 0), (1, 2)]:
        xs = {n: x[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v", "do")}
        one = gpu_grads_dense(xs, True)
        for g_full, g_one in zip(full, one):
            diff = (g_full[b:b + 1, :, h:h + 1].float() - g_one.float()).abs().max().item()
            assert diff <= 2e-2 * max(g_one.float().abs().max().item(), 1e-6)


def test_mid_workload_sampled_heads():
    """Full size (B16 H16 N2048 d64, non-causal); four (b, h) heads in full."""
    w = synth.WORKLOADS["mid"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=w.seed, device="cuda")
    o, lse = ops.fwd(x["q"], x["k"], x["v"])
    dq, dk, dv = ops.bwd(x["q"], x["k"], x["v"], o, lse, x["do"])
    torch.cuda.synchronize()
    for b, h in [(0, 0), (5, 11), (15, 15), (9, 3)]:
        args = [synth.to_f64(x[n][b, :, h]) for n in ("q", "k", "v", "do")]
        ref = oracle.head_backward(*args, w.scale, False)
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert_grad(synth.to_f64(g[b, :, h]), r, f"mid {name} b{b} h{h}")


def test_long_workload_sampled_heads():
    """Full size (B2 H16 N8192 d128, causal, K x3 in heads 0-7); one boosted
    and one plain head in full."""
    w = synth.WORKLOADS["long"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=w.seed, k_boost=w.k_boost, device="cuda")
    o, lse = ops.fwd(x["q"], x["k"], x["v"], causal=True)
    dq, dk, dv = ops.bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True)
    torch.cuda.synchronize()
    for b, h in [(0, 2), (1, 13)]:
        args = [synth.to_f64(x[n][b, :, h]) for n in ("q", "k", "v", "do")]
        ref = oracle.head_backward(*args, w.scale, True)
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert_grad(synth.to_f64(g[b, :, h]), r, f"long {name} b{b} h{h}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward(d, causal):
    lengths = [1, 130, 0, 257, 64, 500]
    x = synth.make_varlen(lengths, 3, d, seed=31)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ops.fwd_varlen(q, k, v, cu.cuda(), max(lengths), causal=causal)
    dq, dk, dv = ops.bwd_varlen(q, k, v, o, lse, do, cu.cuda(), max(lengths), causal=causal)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    ref = oracle.varlen_backward(*(synth.to_f64(x[n]) for n in ("q", "k", "v", "do")), cu.tolist(),
                                 1.0 / np.sqrt(d), causal)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad(synth.to_f64(g), r, f"varlen {name}")


def test_varlen_workload_sampled_sequences():
    """Full size packed batch (32 seeded lengths in [128, 4096], H32 d128,
    causal); three sequences x two heads in full."""
    w = synth.WORKLOADS["varlen"]
    lengths = synth.varlen_lengths(w.B, w.len_lo, w.len_hi, w.seed)
    x = synth.make_varlen(lengths, w.H, w.d, seed=w.seed, device="cuda")
    cu = x["cu_seqlens"].cuda()
    mx = int(lengths.max())
    o, lse = ops.fwd_varlen(x["q"], x["k"], x["v"], cu, mx, causal=True)
    dq, dk, dv = ops.bwd_varlen(x["q"], x["k"], x["v"], o, lse, x["do"], cu, mx, causal=True)
    torch.cuda.synchronize()
    cuh = x["cu_seqlens"].tolist()
    order = np.argsort(lengths.numpy())
    for b in [int(order[0]), int(order[-1]), 12]:
        lo, hi = cuh[b], cuh[b + 1]
        for h in (1, 30):
            args = [synth.to_f64(x[n][lo:hi, h]) for n in ("q", "k", "v", "do")]
            ref = oracle.head_backward(*args, w.scale, True)
            for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
                assert_grad(synth.to_f64(g[lo:hi, h]), r, f"varlen {name} seq{b} h{h}")
