"""Pins of the paged cache's write side (oracle.paged): tokens appended through
the block table read back in order through the (independently pinned) gather;
a page is taken only when the last one fills; shared pages are copied before a
write and never changed under another sequence; released pages come back.
Mutants with a plausible mistake in each rule are rejected."""
import numpy as np
import pytest

from oracle import attention as A
from oracle import paged as PG

RNG = np.random.default_rng(5)
H, D = 2, 3


def tokens(n):
    return RNG.standard_normal((n, H, D))


def check_append_readback(append):
    P, n_pages = 4, 30
    kp, vp = np.zeros((n_pages, P, H, D)), np.zeros((n_pages, P, H, D))
    free = list(range(n_pages))[::-1]
    table, L = [], 0
    ks, vs = tokens(23), tokens(23)
    ok = True
    for i in range(23):
        before = len(free)
        L = append(kp, vp, table, L, ks[i], vs[i], free)
        ok &= len(table) == -(-L // P)                         # at most one partly filled page
        ok &= (before - len(free)) == (1 if i % P == 0 else 0)  # a page only when the last one filled
    ok &= np.array_equal(A.gather_pages(kp, table, L), ks) and np.array_equal(A.gather_pages(vp, table, L), vs)
    return bool(ok)


def mutant_page_per_token(k_pages, v_pages, block_table, seq_len, k, v, free_pages):
    """Takes a fresh page for every token (when one is left)."""
    P = k_pages.shape[1]
    if free_pages:
        block_table.append(free_pages.pop())
    page = block_table[-1]
    k_pages[page, seq_len % P] = k
    v_pages[page, seq_len % P] = v
    return seq_len + 1


def mutant_slot_from_table_length(k_pages, v_pages, block_table, seq_len, k, v, free_pages):
    P = k_pages.shape[1]
    if seq_len % P == 0:
        block_table.append(free_pages.pop())
    page = block_table[-1]
    k_pages[page, len(block_table) % P] = k  # wrong slot
    v_pages[page, len(block_table) % P] = v
    return seq_len + 1


def test_append_token_reads_back():
    assert check_append_readback(PG.append_token)


@pytest.mark.parametrize("mutant", [mutant_page_per_token, mutant_slot_from_table_length])
def test_append_mutants_are_rejected(mutant):
    assert not check_append_readback(mutant)


# ------------------------------------------------------------------ the pool

def run_pool(pool_cls, fork_len=21, P=16):
    """Parent with fork_len tokens; a child forks it, both then append 20
    tokens.  Returns whether every rule held."""
    n_pages = 16
    pool = pool_cls(n_pages, P, 4, 8)
    kp, vp = np.zeros((n_pages, P, H, D)), np.zeros((n_pages, P, H, D))
    parent = pool.add_seq()
    pk, pv = tokens(fork_len + 20), tokens(fork_len + 20)
    for i in range(fork_len):
        PG.apply_append(kp, vp, *pool.reserve_append(parent), pk[i], pv[i])
    child = pool.fork(parent)
    ck, cv = tokens(20), tokens(20)
    copies = 0
    for i in range(20):
        page, slot, src = pool.reserve_append(child)
        copies += src >= 0
        PG.apply_append(kp, vp, page, slot, src, ck[i], cv[i])
        # the parent's view never changes under the child's writes
        tab, lens = pool.block_table()
        if not np.array_equal(A.gather_pages(kp, tab[parent], int(lens[parent])), pk[:fork_len]):
            return False
    for i in range(20):
        page, slot, src = pool.reserve_append(parent)
        copies += src >= 0
        PG.apply_append(kp, vp, page, slot, src, pk[fork_len + i], pv[fork_len + i])
    tab, lens = pool.block_table()
    ok = np.array_equal(A.gather_pages(kp, tab[parent], int(lens[parent])), pk)
    ok &= np.array_equal(A.gather_pages(kp, tab[child], int(lens[child])), np.concatenate([pk[:fork_len], ck]))
    ok &= np.array_equal(A.gather_pages(vp, tab[child], int(lens[child])), np.concatenate([pv[:fork_len], cv]))
    # a copy only when the shared last page was partly filled, and only once
    ok &= copies == (1 if fork_len % P else 0)
    # full pages of the prompt stay shared
    shared = fork_len // P
    ok &= list(tab[parent][:shared]) == list(tab[child][:shared])
    # every page is free or referenced as many times as tables hold it
    held = {}
    for s in (parent, child):
        for p in tab[s][:-(-int(lens[s]) // P)]:
            held[int(p)] = held.get(int(p), 0) + 1
    ok &= all(pool.ref[p] == c for p, c in held.items())
    ok &= sorted(pool.free + list(held)) == list(range(n_pages))
    pool.release(child)
    pool.release(parent)
    ok &= sorted(pool.free) == list(range(n_pages)) and all(r == 0 for r in pool.ref)
    return bool(ok)


@pytest.mark.parametrize("fork_len", [21, 32, 1, 16])
def test_pool_fork_copy_on_write_release(fork_len):
    assert run_pool(PG.PagePool, fork_len)


class MutantNoCopy(PG.PagePool):
    """Writes into a shared page without copying it."""

    def reserve_append(self, s):
        P = self.page_size
        t = self.tables[s]
        L = self.lens[s]
        if L % P == 0:
            t.append(self._take())
        self.lens[s] = L + 1
        return t[-1], L % P, -1


class MutantForkWithoutRefs(PG.PagePool):
    """Forks without counting the shared pages."""

    def fork(self, parent):
        child = self.add_seq()
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        return child


class MutantCopyEveryWrite(PG.PagePool):
    """Copies the last page on every write, shared or not."""

    def reserve_append(self, s):
        P = self.page_size
        t = self.tables[s]
        L = self.lens[s]
        src = -1
        if L % P == 0:
            t.append(self._take())
        else:
            new = self._take()
            self.ref[t[-1]] -= 1
            if self.ref[t[-1]] == 0:
                self.free.append(t[-1])
            src = t[-1]
            t[-1] = new
        self.lens[s] = L + 1
        return t[-1], L % P, src


@pytest.mark.parametrize("mutant", [MutantNoCopy, MutantForkWithoutRefs, MutantCopyEveryWrite])
def test_pool_mutants_are_rejected(mutant):
    assert not all(run_pool(mutant, fl) for fl in (21, 32))


def test_out_of_pages_changes_nothing():
    pool = PG.PagePool(2, 4, 2, 4)
    s = pool.add_seq()
    for _ in range(8):
        pool.reserve_append(s)
    tab, lens = pool.block_table()
    with pytest.raises(PG.OutOfPages):
        pool.reserve_append(s)
    tab2, lens2 = pool.block_table()
    assert np.array_equal(tab, tab2) and np.array_equal(lens, lens2) and pool.free == []


def test_free_list_is_a_stack():
    pool = PG.PagePool(5, 2, 3, 4)
    a, b = pool.add_seq(), pool.add_seq()
    assert [pool.reserve_append(a)[0] for _ in range(3)] == [0, 0, 1]
    assert pool.reserve_append(b)[0] == 2
    pool.release(a)                      # pages 0, 1 pushed in table order
    c = pool.add_seq()
    assert c == 0                        # smallest free slot
    assert pool.reserve_append(c)[0] == 1
