"""A decode loop over a paged cache on the GPU: the host pool reserves slots,
fa_paged_append copies shared pages and writes the tokens, fa_decode_paged
attends.  Page contents must equal the oracle's bit for bit (pure data
movement), outputs the oracle's paged decode within the decode tolerances."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import ops
from oracle import paged as PG
from tests.parity import assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_decode_loop_with_forks(d):
    P, n_pages, max_seqs, max_blocks, Hkv, Hq = 16, 48, 6, 12, 2, 2
    g = torch.Generator().manual_seed(d)
    pool, ref = ops.PagePool(n_pages, P, max_seqs, max_blocks), PG.PagePool(n_pages, P, max_seqs, max_blocks)
    k_pages = torch.zeros((n_pages, P, Hkv, d), dtype=torch.bfloat16, device="cuda")
    v_pages = torch.zeros_like(k_pages)
    rk, rv = np.zeros((n_pages, P, Hkv, d)), np.zeros((n_pages, P, Hkv, d))

    def step(seqs):
        n = len(seqs)
        kn = torch.randn((n, Hkv, d), generator=g).to(torch.bfloat16)
        vn = torch.randn((n, Hkv, d), generator=g).to(torch.bfloat16)
        page, slot, src = pool.reserve_append(seqs)
        ops.paged_append(kn.cuda(), vn.cuda(), k_pages, v_pages, page.cuda(), slot.cuda(), src.cuda())
        for i, s in enumerate(seqs):
            want = ref.reserve_append(s)
            assert (int(page[i]), int(slot[i]), int(src[i])) == want
            PG.apply_append(rk, rv, *want, synth.to_f64(kn[i]), synth.to_f64(vn[i]))

    a, b = pool.add_seq(), pool.add_seq()
    assert (a, b) == (ref.add_seq(), ref.add_seq())
    for _ in range(37):                      # prompts: a gets 37 tokens, b 20
        step([a])
    for _ in range(20):
        step([b])
    c = pool.fork(a)                         # shares a's 37-token prompt (last page partly filled)
    assert c == ref.fork(a)
    for t in range(30):                      # decode: every sequence one token per step
        step([a, b, c] if t % 3 else [c, a, b])
        if t == 12:
            pool.release(b)
            ref.release(b)
            b = pool.add_seq()
            assert b == ref.add_seq()
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert np.array_equal(synth.to_f64(k_pages), rk) and np.array_equal(synth.to_f64(v_pages), rv)

    table, lens = pool.export()
    live = [a, b, c]
    q = torch.randn((len(live), 1, Hq, d), generator=g).to(torch.bfloat16)
    bt = table[live].contiguous()
    sl = lens[live].contiguous()
    o, lse = ops.decode_paged(q.cuda(), k_pages, v_pages, bt.cuda(), sl.cuda(), int(sl.max()))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.paged_decode_forward(synth.to_f64(q), rk, rv, bt.numpy(), sl.tolist(), 1 / math.sqrt(d))
    assert_o(synth.to_f64(o), o_ref, f"paged loop d{d}")
    assert_lse(lse.cpu().numpy(), l_ref, f"paged loop d{d}")


def test_append_rejects_a_page_outside_the_pool():
    d, P, n_pages = 64, 4, 3
    k_pages = torch.zeros((n_pages, P, 1, d), dtype=torch.bfloat16, device="cuda")
    v_pages = torch.zeros_like(k_pages)
    kn = torch.ones((1, 1, d), dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([7], dtype=torch.int32, device="cuda")
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_append(kn, kn, k_pages, v_pages, bad, zero, zero - 1)
    torch.cuda.synchronize()
    assert ops.device_error() == 0x2000
    assert torch.all(k_pages == 0)
