"""The library's host page pool (fa_pool_*) against the oracle's pool: the same
operations give the same block tables, lengths, reference counts and free
pages, and a batch that does not fit changes nothing."""
import numpy as np
import pytest

from exact_attention_94_gb300 import _lib, build, ops
from oracle import paged as PG


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def same(pool, ref):
    tab, lens = pool.export()
    rtab, rlens = ref.block_table()
    assert np.array_equal(tab.numpy(), rtab) and np.array_equal(lens.numpy(), rlens)
    assert pool.free_pages() == len(ref.free)
    assert all(pool.refcount(p) == ref.ref[p] for p in range(len(ref.ref)))


def test_random_operations_match_the_oracle():
    rng = np.random.default_rng(3)
    n_pages, P, max_seqs, max_blocks = 40, 4, 6, 12
    pool, ref = ops.PagePool(n_pages, P, max_seqs, max_blocks), PG.PagePool(n_pages, P, max_seqs, max_blocks)
    live = []
    for step in range(400):
        r = rng.random()
        if (r < 0.08 or not live) and len(live) < max_seqs:
            s = pool.add_seq()
            assert s == ref.add_seq()
            live.append(s)
        elif r < 0.14 and len(live) < max_seqs:
            parent = int(rng.choice(live))
            c = pool.fork(parent)
            assert c == ref.fork(parent)
            live.append(c)
        elif r < 0.2 and len(live) > 1:
            s = int(rng.choice(live))
            pool.release(s)
            ref.release(s)
            live.remove(s)
        else:
            batch = [int(x) for x in rng.permutation(live)[: rng.integers(1, len(live) + 1)]]
            # only batches that fit the tables (the oracle raises on a full table)
            if any(ref.lens[s] % P == 0 and len(ref.tables[s]) >= max_blocks for s in batch):
                continue
            try:
                page, slot, src = pool.reserve_append(batch)
            except _lib.FaError as e:
                assert e.status == _lib.FA_ERR_OUT_OF_PAGES
                same(pool, ref)  # nothing changed
                # the oracle agrees that the batch does not fit
                snapshot = (list(ref.free), list(ref.ref), [list(t) if t is not None else None for t in ref.tables],
                            list(ref.lens))
                with pytest.raises(PG.OutOfPages):
                    for s in batch:
                        ref.reserve_append(s)
                ref.free, ref.ref, ref.tables, ref.lens = snapshot
                continue
            want = [ref.reserve_append(s) for s in batch]
            assert [tuple(int(t[i]) for t in (page, slot, src)) for i in range(len(batch))] == want
        same(pool, ref)


def test_two_sharers_in_one_batch_need_one_page():
    """A page held twice and written by both holders in one batch is copied
    once (the second writer is then its last holder): one free page suffices."""
    pool = ops.PagePool(2, 4, 2, 4)
    a = pool.add_seq()
    pool.reserve_append([a])                 # page 0, slot 0
    b = pool.fork(a)                         # page 0 shared
    assert pool.free_pages() == 1
    page, slot, src = pool.reserve_append([a, b])
    assert page.tolist() == [1, 0] and slot.tolist() == [1, 1] and src.tolist() == [0, -1]
    assert pool.refcount(0) == 1 and pool.refcount(1) == 1 and pool.free_pages() == 0


def test_batch_that_does_not_fit_changes_nothing():
    pool = ops.PagePool(3, 2, 3, 4)
    s = [pool.add_seq() for _ in range(3)]
    pool.reserve_append(s)                   # three pages taken
    pool.reserve_append(s)                   # second slots
    before = pool.export()
    with pytest.raises(_lib.FaError) as e:
        pool.reserve_append(s)
    assert e.value.status == _lib.FA_ERR_OUT_OF_PAGES
    after = pool.export()
    assert all(np.array_equal(x.numpy(), y.numpy()) for x, y in zip(before, after))


def test_bad_requests():
    pool = ops.PagePool(4, 2, 2, 1)
    a = pool.add_seq()
    with pytest.raises(_lib.FaError):
        pool.reserve_append([a, a])          # repeated sequence
    with pytest.raises(_lib.FaError):
        pool.reserve_append([1])             # not a live sequence
    pool.reserve_append([a])
    pool.reserve_append([a])
    with pytest.raises(_lib.FaError):
        pool.reserve_append([a])             # table full (max_blocks = 1)
    lib = ops.lib()
    assert not lib.fa_pool_create(0, 16, 1, 1)
    assert lib.fa_pool_free_pages(None) == -1
