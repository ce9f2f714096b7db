"""Grouped-query attention on the GPU against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import ops
from tests.parity import assert_grad, assert_lse, assert_o

pytestmark = pytest.mark.gpu


def make(B, N, Hq, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda H: torch.randn((B, N, H, d), generator=g).to(torch.bfloat16)
    return {"q": mk(Hq), "k": mk(Hkv), "v": mk(Hkv), "do": mk(Hq)}


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Hq,Hkv", [(300, 8, 2), (257, 6, 3), (640, 4, 1)])
def test_gqa_forward_backward(d, causal, N, Hq, Hkv):
    x = make(2, N, Hq, Hkv, d, seed=N + Hq)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ops.fwd_gqa(q, k, v, causal=causal)
    dq, dk, dv = ops.bwd_gqa(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    f64 = {n: synth.to_f64(x[n]) for n in x}
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.gqa_forward(f64["q"], f64["k"], f64["v"], scale, causal)
    assert_o(synth.to_f64(o), o_ref, "gqa O")
    assert_lse(lse.cpu().numpy(), l_ref, "gqa lse")
    refs = oracle.gqa_backward(f64["q"], f64["k"], f64["v"], f64["do"], scale, causal)
    for name, gg, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert_grad(synth.to_f64(gg), r, f"gqa {name}")


def test_gqa_with_group_one_matches_plain_calls():
    x = make(1, 384, 4, 4, 128, seed=3)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o1, l1 = ops.fwd_gqa(q, k, v, causal=True)
    o2, l2 = ops.fwd(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 1), (12, 4)])
def test_gqa_decode(Hq, Hkv):
    B, L, d = 3, 1000, 128
    g = torch.Generator().manual_seed(Hq + Hkv)
    q = torch.randn((B, 1, Hq, d), generator=g).to(torch.bfloat16)
    kc = torch.randn((B, L, Hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, L, Hkv, d), generator=g).to(torch.bfloat16)
    o, lse = ops.decode_gqa(q.cuda(), kc.cuda(), vc.cuda())
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    o_ref, l_ref = oracle.gqa_decode_forward(synth.to_f64(q), synth.to_f64(kc), synth.to_f64(vc), 1 / math.sqrt(d))
    assert_o(synth.to_f64(o), o_ref, "gqa decode O")
    assert_lse(lse.cpu().numpy(), l_ref, "gqa decode lse")
