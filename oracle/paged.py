"""Reference for the write side of the paged KV cache: appending a token, the
free list, and sharing pages between sequences.

TEST INFRASTRUCTURE ONLY, like ``oracle.attention``: imported by ``tests/``
and never by the library.

Source: zerotofrontier.app "efficient-attention/flash-2-3", section "Paged KV
caches, a preview of serving": the cache is a pool of fixed-size pages (16
tokens by default); each sequence's block table maps its logical blocks
(tokens 0-15, 16-31, ...) to physical pages; a new page is taken from the free
list only when the sequence's last page fills, so at most one partly filled
page per sequence is wasted; sequences that share a prompt share its pages
and copy one only when they would write to it.  The page prints a stub
``append_token(k_pages, v_pages, block_table, seq_len, k, v, free_pages)``.

Readings (the page leaves them open):
  * the free list is a stack: pages start as [n-1, ..., 1, 0], a page is taken
    from the end (page 0 first) and a released page is pushed on the end;
  * a write into a shared page (reference count > 1) first copies it to a page
    taken from the free list; only a sequence's last page can be written, so
    only it is ever copied;
  * sequence slots are reused: a new sequence takes the smallest free slot;
  * running out of pages is an error, reported before anything changes.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import numpy as np


class OutOfPages(RuntimeError):
    pass


def append_token(k_pages, v_pages, block_table: List[int], seq_len: int, k, v, free_pages: List[int]) -> int:
    """The page's single-sequence step: write k, v ([H, d]) as token seq_len,
    taking a page from ``free_pages`` when the last one is full (or there is
    none).  Modifies the pages and the table in place; returns the new length."""
    P = k_pages.shape[1]
    if seq_len % P == 0:
        if not free_pages:
            raise OutOfPages("no free page")
        block_table.append(free_pages.pop())
    page = block_table[seq_len // P]
    k_pages[page, seq_len % P] = k
    v_pages[page, seq_len % P] = v
    return seq_len + 1


class PagePool:
    """Block tables, lengths and reference counts of up to ``max_seqs``
    sequences over ``num_pages`` pages of ``page_size`` tokens."""

    def __init__(self, num_pages: int, page_size: int, max_seqs: int, max_blocks: int):
        self.page_size = page_size
        self.max_blocks = max_blocks
        self.free = list(range(num_pages))[::-1]
        self.ref = [0] * num_pages
        self.tables: List[Optional[List[int]]] = [None] * max_seqs
        self.lens = [0] * max_seqs

    def _take(self) -> int:
        if not self.free:
            raise OutOfPages("no free page")
        p = self.free.pop()
        self.ref[p] = 1
        return p

    def add_seq(self) -> int:
        for s, t in enumerate(self.tables):
            if t is None:
                self.tables[s] = []
                self.lens[s] = 0
                return s
        raise RuntimeError("no free sequence slot")

    def fork(self, parent: int) -> int:
        """A new sequence sharing every page of ``parent`` (a common prompt)."""
        child = self.add_seq()
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for p in self.tables[child]:
            self.ref[p] += 1
        return child

    def release(self, s: int) -> None:
        for p in self.tables[s]:
            self.ref[p] -= 1
            if self.ref[p] == 0:
                self.free.append(p)
        self.tables[s] = None
        self.lens[s] = 0

    def reserve_append(self, s: int) -> Tuple[int, int, int]:
        """Prepare the write of token lens[s]: returns (page, slot, copy_src),
        copy_src >= 0 when the page must first receive a copy of copy_src."""
        P = self.page_size
        t = self.tables[s]
        L = self.lens[s]
        copy_src = -1
        if L % P == 0:
            if len(t) >= self.max_blocks:
                raise RuntimeError("block table full")
            t.append(self._take())
        elif self.ref[t[-1]] > 1:
            new = self._take()
            self.ref[t[-1]] -= 1
            copy_src = t[-1]
            t[-1] = new
        self.lens[s] = L + 1
        return t[-1], L % P, copy_src

    def block_table(self) -> Tuple[np.ndarray, np.ndarray]:
        """[max_seqs, max_blocks] int32 (unused entries 0) and lengths [max_seqs]."""
        tab = np.zeros((len(self.tables), self.max_blocks), dtype=np.int32)
        for s, t in enumerate(self.tables):
            if t:
                tab[s, :len(t)] = t
        return tab, np.array(self.lens, dtype=np.int32)


def apply_append(k_pages, v_pages, page: int, slot: int, copy_src: int, k, v) -> None:
    """The device side of one append: the copy (if any), then the write."""
    if copy_src >= 0:
        k_pages[page] = k_pages[copy_src]
        v_pages[page] = v_pages[copy_src]
    k_pages[page, slot] = k
    v_pages[page, slot] = v
