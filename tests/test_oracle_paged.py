"""Pins of the oracle's paged-cache decode: the test itself scatters each
sequence's own cache into a shuffled page pool (independently of the oracle's
gather), and the paged decode must equal plain decode over each sequence."""
import numpy as np
import pytest

from oracle import attention as A

RNG = np.random.default_rng(77)


def scatter(caches, page_size, spare=2):
    """Place each sequence's [L_b, H, d] cache into pages of a shuffled pool."""
    H, d = caches[0].shape[1:]
    blocks = [-(-len(c) // page_size) for c in caches]
    n_pages = sum(blocks) + spare
    pool = RNG.standard_normal((n_pages, page_size, H, d)) * 7.0  # unused slots hold large junk
    order = RNG.permutation(n_pages)
    table = np.zeros((len(caches), max(1, max(blocks))), dtype=np.int64)
    nxt = 0
    for b, c in enumerate(caches):
        for j in range(blocks[b]):
            page = order[nxt]
            nxt += 1
            table[b, j] = page
            seg = c[j * page_size:(j + 1) * page_size]
            pool[page, :len(seg)] = seg
    return pool, table


@pytest.mark.parametrize("page_size", [4, 16])
def test_paged_equals_per_sequence_decode(page_size):
    lengths = [1, 15, 16, 17, 40]
    H, d = 3, 5
    ks = [RNG.standard_normal((L, H, d)) for L in lengths]
    vs = [RNG.standard_normal((L, H, d)) for L in lengths]
    k_pool, table = scatter(ks, page_size)
    v_pool = np.zeros_like(k_pool)
    # same placement for V: reuse the table
    for b, c in enumerate(vs):
        for j in range(-(-len(c) // page_size)):
            seg = c[j * page_size:(j + 1) * page_size]
            v_pool[table[b, j], :len(seg)] = seg
    q = RNG.standard_normal((len(lengths), 1, H, d))
    o, lse = A.paged_decode_forward(q, k_pool, v_pool, table, lengths, 0.4)
    for b, L in enumerate(lengths):
        for h in range(H):
            oh, lh = A.head_forward(q[b, :, h], ks[b][:, h], vs[b][:, h], 0.4, False)
            assert np.max(np.abs(o[b, 0, h] - oh[0])) < 1e-12
            assert abs(lse[b, h] - lh[0]) < 1e-12


def test_contiguous_pages_equal_contiguous_decode():
    B, L, H, d, P = 2, 32, 2, 4, 8
    k = RNG.standard_normal((B, L, H, d))
    v = RNG.standard_normal((B, L, H, d))
    q = RNG.standard_normal((B, 1, H, d))
    k_pool = k.reshape(B * L // P, P, H, d)
    v_pool = v.reshape(B * L // P, P, H, d)
    table = np.arange(B * L // P).reshape(B, L // P)
    o1, l1 = A.paged_decode_forward(q, k_pool, v_pool, table, [L] * B, 0.3)
    o2, l2 = A.decode_forward(q, k, v, 0.3)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13


def mutant_gather_keeps_garbage(pages, block_table_row, seq_len):
    # the "gather" stub: whole pages, unused slots included
    n_blocks = -(-seq_len // pages.shape[1])
    return np.concatenate([pages[int(block_table_row[j])] for j in range(n_blocks)], axis=0)


def test_gather_keeping_garbage_slots_is_rejected(monkeypatch):
    lengths = [5, 17]
    H, d = 2, 3
    ks = [RNG.standard_normal((L, H, d)) for L in lengths]
    pool, table = scatter(ks, 8)
    q = RNG.standard_normal((2, 1, H, d))
    monkeypatch.setattr(A, "gather_pages", mutant_gather_keeps_garbage)
    o, _ = A.paged_decode_forward(q, pool, pool, table, lengths, 0.5)
    ok = True
    for b in range(2):
        for h in range(H):
            oh, _ = A.head_forward(q[b, :, h], ks[b][:, h], ks[b][:, h], 0.5, False)
            ok &= np.max(np.abs(o[b, 0, h] - oh[0])) < 1e-9
    assert not ok
