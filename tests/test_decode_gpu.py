"""Split-KV decode parity: final O and lse against the float64 oracle (dense
single-query attention over the whole cache), and the split step's partial
results against the oracle's own split step."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import ops
from tests.parity import assert_lse, assert_o

pytestmark = pytest.mark.gpu


def run_decode(B, H, L, d, num_splits, seed=0):
    x = synth.make_decode(B, H, L, d, seed=seed)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ops.decode(q, k, v, num_splits=num_splits)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    return x, o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [1, 3, 4, 5, 127, 1000])
@pytest.mark.parametrize("num_splits", [0, 1, 2, 7])
def test_decode_small(d, L, num_splits):
    if num_splits > L:
        pytest.skip("more splits than keys")
    B, H = 3, 4
    x, o, lse = run_decode(B, H, L, d, num_splits, seed=L)
    o_ref, l_ref = oracle.decode_forward(*(synth.to_f64(x[n]) for n in ("q", "k", "v")), 1.0 / math.sqrt(d))
    assert_o(synth.to_f64(o), o_ref, f"decode O L{L} d{d} S{num_splits}")
    assert_lse(lse.cpu().numpy(), l_ref, f"decode lse L{L} d{d} S{num_splits}")


@pytest.mark.parametrize("H", [40, 64, 7])
def test_decode_head_groups(H):
    """H = 40 runs in groups of 20 heads, H = 64 in two groups of 32, H = 7 in one."""
    x, o, lse = run_decode(2, H, 600, 128, 3, seed=H)
    o_ref, l_ref = oracle.decode_forward(*(synth.to_f64(x[n]) for n in ("q", "k", "v")), 1.0 / math.sqrt(128))
    assert_o(synth.to_f64(o), o_ref, f"decode H{H}")
    assert_lse(lse.cpu().numpy(), l_ref, f"decode H{H}")


def test_decode_partials_match_oracle_split_step():
    """The workspace after a call holds each chunk's normalised output and its
    log-sum-exp (base 2); they equal the oracle's split step on the same
    chunk bounds."""
    B, H, L, d, S = 2, 3, 301, 128, 4
    x = synth.make_decode(B, H, L, d, seed=5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    nbytes = ops.lib().fa_decode_workspace_bytes(B, H, d, S)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ops.decode(q, k, v, num_splits=S, workspace=ws)
    torch.cuda.synchronize()
    part_o = ws[: B * H * S * d * 4].view(torch.float32).view(B, H, S, d).cpu().numpy()
    off = (B * H * S * d * 4 + 255) // 256 * 256
    part_l2 = ws[off: off + B * H * S * 4].view(torch.float32).view(B, H, S).cpu().numpy()
    ref_o, ref_l = oracle.decode_partials(*(synth.to_f64(x[n]) for n in ("q", "k", "v")), 1.0 / math.sqrt(d), S)
    assert np.max(np.abs(part_o - ref_o)) < 2e-3
    assert np.max(np.abs(part_l2 * math.log(2.0) - ref_l)) < 1e-3


def test_decode_empty_cache():
    """L = 0: every row is fully masked -> O = 0 and lse = -inf."""
    q = torch.randn(2, 1, 3, 128, device="cuda").to(torch.bfloat16)
    kv = torch.empty(2, 0, 3, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = ops.decode(q, kv, kv, num_splits=1)
    torch.cuda.synchronize()
    assert torch.all(o == 0)
    assert torch.all(torch.isneginf(lse))


def test_decode_workload_sampled_heads():
    """Full size (B64 L32768 H32 d128; 34.4 GB of cache generated on the
    device); six (b, h) pairs compared with the oracle over the whole cache."""
    w = synth.WORKLOADS["decode"]
    x = synth.make_decode(w.B, w.H, w.N, w.d, seed=w.seed, device="cuda")
    o, lse = ops.decode(x["q"], x["k"], x["v"])
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    for b, h in [(0, 0), (7, 31), (33, 12), (63, 5), (20, 20), (63, 31)]:
        qh = synth.to_f64(x["q"][b, :, h])
        kh, vh = synth.to_f64(x["k"][b, :, h]), synth.to_f64(x["v"][b, :, h])
        oh, lh = oracle.head_forward(qh, kh, vh, w.scale, False)
        assert_o(synth.to_f64(o[b, 0, h]), oh[0], f"decode b{b} h{h}")
        assert_lse(lse[b, h].cpu().numpy(), lh[0], f"decode b{b} h{h}")
    del x
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- paged KV cache

def run_paged(lengths, H, d, page_size, num_splits, seed=0):
    x = synth.make_paged_decode(lengths, H, d, page_size=page_size, seed=seed)
    dev = {n: x[n].cuda() for n in x}
    o, lse = ops.decode_paged(dev["q"], dev["k_pages"], dev["v_pages"], dev["block_table"], dev["seq_lens"],
                              max(lengths), num_splits=num_splits)
    torch.cuda.synchronize()
    return x, o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("page_size", [16, 32])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_paged_decode_ragged(d, page_size, num_splits):
    lengths = [1, 15, 16, 17, 100, 1000]
    x, o, lse = run_paged(lengths, 4, d, page_size, num_splits, seed=page_size)
    assert ops.device_error() == 0
    o_ref, l_ref = oracle.paged_decode_forward(synth.to_f64(x["q"]), synth.to_f64(x["k_pages"]),
                                               synth.to_f64(x["v_pages"]), x["block_table"].numpy(),
                                               x["seq_lens"].tolist(), 1.0 / math.sqrt(d))
    assert_o(synth.to_f64(o), o_ref, f"paged O d{d} P{page_size} S{num_splits}")
    assert_lse(lse.cpu().numpy(), l_ref, f"paged lse d{d} P{page_size} S{num_splits}")


def test_paged_in_order_equals_contiguous_decode():
    """Pages laid out in order with full lengths give the contiguous path's bits."""
    B, H, L, d, P = 3, 8, 512, 128, 16
    x = synth.make_decode(B, H, L, d, seed=21)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    table = torch.arange(B * L // P, dtype=torch.int32, device="cuda").view(B, L // P)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    o1, l1 = ops.decode(q, k, v, num_splits=4)
    o2, l2 = ops.decode_paged(q, k.view(B * L // P, P, H, d), v.view(B * L // P, P, H, d), table, lens, L,
                              num_splits=4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paged_bad_table_entry_is_reported_not_read():
    lengths = [40, 20]
    x = synth.make_paged_decode(lengths, 2, 64, page_size=16, seed=5)
    bt = x["block_table"].clone()
    bt[1, 0] = 10_000_000  # far outside the pool
    dev = {n: x[n].cuda() for n in x}
    ops.decode_paged(dev["q"], dev["k_pages"], dev["v_pages"], bt.cuda(), dev["seq_lens"], max(lengths))
    torch.cuda.synchronize()
    assert ops.device_error() == 0x2000
    assert ops.device_error() == 0


# ---------------------------------------------------------------- sliding window, grouped heads

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("wl", [0, 5, 127, 300, 5000, -1])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_window(d, wl, num_splits):
    """Keys len-1-wl .. len-1 only; against the masked oracle with one query."""
    B, Hq, Hkv, L = 3, 8, 2, 1000
    g = torch.Generator().manual_seed(wl + 7 + d)
    q = torch.randn((B, 1, Hq, d), generator=g).to(torch.bfloat16)
    kc = torch.randn((B, L, Hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, L, Hkv, d), generator=g).to(torch.bfloat16)
    span = L if wl < 0 or wl >= L else wl + 1
    if num_splits > span:
        pytest.skip("more splits than keys in the window")
    o, lse = ops.decode_window(q.cuda(), kc.cuda(), vc.cuda(), wl, num_splits=num_splits)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    o_ref, l_ref = oracle.masked_forward(synth.to_f64(q), synth.to_f64(kc), synth.to_f64(vc), 1 / math.sqrt(d), wl, 0)
    assert_o(synth.to_f64(o), o_ref, f"window decode wl{wl}")
    assert_lse(lse.cpu().numpy(), l_ref[:, :, 0], f"window decode wl{wl}")


@pytest.mark.parametrize("wl", [-1, 40, 17])
def test_paged_decode_window_grouped(wl):
    """Ragged paged caches, 4 query heads per K/V head, a window."""
    lengths = [1, 15, 16, 17, 100, 1000]
    Hq, Hkv, d, P = 8, 2, 128, 16
    x = synth.make_paged_decode(lengths, Hkv, d, page_size=P, seed=wl + 50)
    g = torch.Generator().manual_seed(wl + 51)
    q = torch.randn((len(lengths), 1, Hq, d), generator=g).to(torch.bfloat16)
    dev = {n: x[n].cuda() for n in x}
    o, lse = ops.decode_paged_window(q.cuda(), dev["k_pages"], dev["v_pages"], dev["block_table"], dev["seq_lens"],
                                     max(lengths), wl, num_splits=3)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    kp, vp = synth.to_f64(x["k_pages"]), synth.to_f64(x["v_pages"])
    for b, Lb in enumerate(lengths):
        kb = oracle.gather_pages(kp, x["block_table"][b].numpy(), Lb)[None]
        vb = oracle.gather_pages(vp, x["block_table"][b].numpy(), Lb)[None]
        o_ref, l_ref = oracle.masked_forward(synth.to_f64(q[b:b + 1]), kb, vb, 1 / math.sqrt(d), wl, 0)
        assert_o(synth.to_f64(o[b:b + 1]), o_ref, f"paged window b{b}")
        assert_lse(lse[b:b + 1].cpu().numpy(), l_ref[:, :, 0], f"paged window b{b}")
