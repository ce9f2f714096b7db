"""Split-KV decode parity: final O and lse against the float64 oracle (dense
single-query attention over the whole cache), and the split step's partial
results against the oracle's own split step."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import _lib, ops
from tests.parity import LSE_TOL, O_TOL, assert_lse, assert_o

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
    B, H = 3, 4
    if num_splits > L:  # more splits than keys: refused before any launch
        x = synth.make_decode(B, H, L, d, seed=L)
        with pytest.raises(_lib.FaError) as e:
            ops.decode(*(x[n].cuda() for n in ("q", "k", "v")), num_splits=num_splits)
        assert e.value.status == _lib.FA_ERR_INVALID_ARG
        return
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
    if num_splits > span:  # more splits than keys in the window: refused before any launch
        with pytest.raises(_lib.FaError) as e:
            ops.decode_window(q.cuda(), kc.cuda(), vc.cuda(), wl, num_splits=num_splits)
        assert e.value.status == _lib.FA_ERR_INVALID_ARG
        return
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


# ---------------------------------------------------------------- decode against the dense path
#
# "Decoding needs a different split" (efficient-attention/flash-2-3): the
# split-KV decode computes the same single-query attention as the dense path,
# only partitioned along the keys and merged.  Each case below runs the dense
# masked forward with one query (N_q = 1, bottom-right aligned, so the query
# sits at the last key) on the same cache and compares the two results within
# the parity tolerances.

def _dense_one_query(q, k, v, window_left=-1):
    """fa_fwd_masked with N_q = 1 over a contiguous cache [B, L, Hkv, d]."""
    o, lse = ops.fwd_masked(q, k, v, window=(window_left, -1))
    return o, lse[:, :, 0]


def _close(o_dec, l_dec, o_den, l_den, what):
    do = (o_dec.double() - o_den.double()).abs().max().item()
    dl = (l_dec - l_den).abs().max().item()
    assert do <= O_TOL, f"{what}: max |O_decode - O_dense| {do:.3e}"
    assert dl <= LSE_TOL, f"{what}: max |lse_decode - lse_dense| {dl:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L,num_splits", [(1, 1), (129, 0), (1000, 3), (4096, 0), (4097, 7)])
def test_decode_equals_dense_path(d, L, num_splits):
    B, H = 3, 8
    x = synth.make_decode(B, H, L, d, seed=L + d)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = ops.decode(q, k, v, num_splits=num_splits)
    o2, l2 = _dense_one_query(q, k, v)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _close(o1, l1, o2, l2, f"decode L{L} d{d} S{num_splits}")


@pytest.mark.parametrize("Hq,Hkv,wl", [(32, 8, -1), (16, 1, -1), (12, 4, 300), (8, 2, 0)])
def test_decode_gqa_window_equals_dense_path(Hq, Hkv, wl):
    B, L, d = 2, 2000, 128
    g = torch.Generator().manual_seed(Hq * 10 + Hkv + wl)
    q = torch.randn((B, 1, Hq, d), generator=g).to(torch.bfloat16).cuda()
    kc = torch.randn((B, L, Hkv, d), generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn((B, L, Hkv, d), generator=g).to(torch.bfloat16).cuda()
    if wl < 0:
        o1, l1 = ops.decode_gqa(q, kc, vc)
    else:
        o1, l1 = ops.decode_window(q, kc, vc, wl)
    o2, l2 = _dense_one_query(q, kc, vc, wl)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _close(o1, l1, o2, l2, f"decode Hq{Hq} Hkv{Hkv} wl{wl}")


@pytest.mark.parametrize("Hq,Hkv,wl", [(4, 4, -1), (8, 2, -1), (8, 2, 40)])
def test_paged_decode_equals_dense_path(Hq, Hkv, wl):
    """Each sequence's pages gathered into a contiguous cache on the device
    (plain indexing), then the dense one-query forward on it."""
    lengths = [1, 15, 16, 17, 100, 1000]
    d, P = 128, 16
    x = synth.make_paged_decode(lengths, Hkv, d, page_size=P, seed=Hq + Hkv + wl)
    g = torch.Generator().manual_seed(Hq + 3 * Hkv + wl)
    q = torch.randn((len(lengths), 1, Hq, d), generator=g).to(torch.bfloat16).cuda()
    dev = {n: x[n].cuda() for n in x}
    o1, l1 = ops.decode_paged_window(q, dev["k_pages"], dev["v_pages"], dev["block_table"], dev["seq_lens"],
                                     max(lengths), wl, num_splits=3)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    for b, Lb in enumerate(lengths):
        pages = dev["block_table"][b, : (Lb + P - 1) // P].long()
        kb = dev["k_pages"][pages].reshape(-1, Hkv, d)[:Lb][None].contiguous()
        vb = dev["v_pages"][pages].reshape(-1, Hkv, d)[:Lb][None].contiguous()
        o2, l2 = _dense_one_query(q[b:b + 1], kb, vb, wl)
        _close(o1[b:b + 1], l1[b:b + 1], o2, l2, f"paged b{b} L{Lb} wl{wl}")
