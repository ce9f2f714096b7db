"""Packed variable-length forward parity against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import ops
from tests.parity import assert_lse, assert_o

pytestmark = pytest.mark.gpu


def check_varlen_fwd(lengths, H, d, causal, seed=0):
    x = synth.make_varlen(lengths, H, d, seed=seed, with_do=False)
    cu = x["cu_seqlens"]
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ops.fwd_varlen(q, k, v, cu.cuda(), max(lengths), causal=causal)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    o_ref, l_ref = oracle.varlen_forward(synth.to_f64(x["q"]), synth.to_f64(x["k"]), synth.to_f64(x["v"]),
                                         cu.tolist(), 1.0 / np.sqrt(d), causal)
    assert_o(synth.to_f64(o), o_ref, f"varlen O {lengths}")
    assert_lse(lse.cpu().numpy(), l_ref, f"varlen lse {lengths}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_ragged(d, causal):
    check_varlen_fwd([1, 5, 128, 129, 300, 700, 17], 3, d, causal, seed=2)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_with_empty_sequence(causal):
    check_varlen_fwd([200, 0, 64, 0, 385], 2, 128, causal, seed=4)


def test_varlen_equals_dense_per_sequence():
    """Each packed sequence equals the dense call on that sequence alone."""
    lengths = [300, 1000, 96]
    x = synth.make_varlen(lengths, 4, 128, seed=9, with_do=False)
    cu = x["cu_seqlens"].tolist()
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ops.fwd_varlen(q, k, v, x["cu_seqlens"].cuda(), max(lengths), causal=True)
    for b, L in enumerate(lengths):
        sl = slice(cu[b], cu[b + 1])
        od, ld = ops.fwd(q[sl].unsqueeze(0).contiguous(), k[sl].unsqueeze(0).contiguous(),
                         v[sl].unsqueeze(0).contiguous(), causal=True)
        assert torch.equal(od[0], o[sl])
        assert torch.equal(ld[0], lse[:, sl])


def test_varlen_workload_sampled_sequences():
    """Full size: 32 sequences with seeded lengths in [128, 4096], H32 d128,
    causal; five sequences compared in full on four heads each."""
    w = synth.WORKLOADS["varlen"]
    lengths = synth.varlen_lengths(w.B, w.len_lo, w.len_hi, w.seed)
    x = synth.make_varlen(lengths, w.H, w.d, seed=w.seed, with_do=False, device="cuda")
    cu = x["cu_seqlens"].tolist()
    o, lse = ops.fwd_varlen(x["q"], x["k"], x["v"], x["cu_seqlens"].cuda(), int(lengths.max()), causal=True)
    torch.cuda.synchronize()
    order = np.argsort(lengths.numpy())
    for b in [int(order[0]), int(order[-1]), 3, 17, 31]:
        lo, hi = cu[b], cu[b + 1]
        for h in (0, 9, 22, 31):
            qh, kh, vh = (synth.to_f64(x[n][lo:hi, h]) for n in ("q", "k", "v"))
            oh, lh = oracle.head_forward(qh, kh, vh, w.scale, True)
            assert_o(synth.to_f64(o[lo:hi, h]), oh, f"varlen seq{b} h{h}")
            assert_lse(lse[h, lo:hi].cpu().numpy(), lh, f"varlen seq{b} h{h}")


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_max_seqlen_too_small_is_reported(which):
    """A sequence longer than the declared max_seqlen would leave rows of it
    uncomputed: the kernels report it (code 0x2001, FA_ERR_INVALID_ARG) and
    write nothing for that sequence instead."""
    lengths = [100, 600, 50]
    x = synth.make_varlen(lengths, 2, 128, seed=6)
    cu = x["cu_seqlens"].cuda()
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ops.fwd_varlen(q, k, v, cu, max(lengths), causal=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    if which == "fwd":
        ops.fwd_varlen(q, k, v, cu, 256, causal=True)
    else:
        ops.bwd_varlen(q, k, v, o, lse, do, cu, 256, causal=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0x2001
    assert ops.device_error() == 0
