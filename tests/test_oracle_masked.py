"""Pins of the masked-attention oracle (causal / sliding window, Nq != Nk).

Each check takes the implementation under test as an argument so that the
mutation tests at the bottom can plant a plausible mistake in a copy of the
oracle and show that a pin rejects it.  The facts pinned come from outside the
masked oracle: the block mask the pages print for a 64-token window, the
pages' 4-queries-against-128-keys example, the square causal oracle (where
both alignments agree), unmasked attention over an explicit slice of keys,
pure-Python brute force, and finite differences.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A
from oracle import masked as M
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(4321)


def rnd(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def fwd_with(visible_fn):
    """masked head forward built on a given visibility function."""
    def f(q, k, v, scale, wl, wr):
        return M.head_forward_visible(q, k, v, scale, visible_fn(len(q), len(k), wl, wr))
    return f


# ------------------------------------------------------------------ checks

def check_block_mask_golden(visible_fn):
    """The pages' printed block mask: a 64-token causal window visits the
    diagonal 128 x 128 tiles and the ones just below them, nothing else.
    Both readings of "64-token window" (64 keys including the query, or 64
    before it) give that pattern."""
    g = json.load(open(os.path.join(GOLDEN, "pages_worked_numbers.json")))["window_64_block_mask"]
    n, t = 1024, g["tile"]
    for wl in (g["window_tokens"] - 1, g["window_tokens"]):
        bm = M.block_mask(visible_fn(n, n, wl, 0), t)
        a, b = np.nonzero(bm)
        if sorted(set((b - a).tolist())) != sorted(g["visited_offsets"]):
            return False
        if bm.sum() != 2 * (n // t) - 1:
            return False
    return True


def check_bottom_right_example(visible_fn):
    """The pages' example: 4 new queries against 128 keys.  Top-left lets the
    first query see key 0 only; the bottom-right convention lets it see every
    key up to its own position, 124, and the last query sees all 128."""
    g = json.load(open(os.path.join(GOLDEN, "pages_worked_numbers.json")))["top_left_causal"]
    nq, nk = g["n_q"], g["n_k"]
    tl = M.top_left_causal_visible(nq, nk)
    if list(np.nonzero(tl[0])[0]) != g["first_query_visible_keys_top_left"]:
        return False
    br = visible_fn(nq, nk, -1, 0)
    return list(np.nonzero(br[0])[0]) == list(range(nk - nq + 1)) and bool(br[-1].all())


def check_square_causal_matches(fwd):
    """Nq == Nk with the window (-1, 0) is plain causal attention, computed by
    the square oracle's own mask; (-1, -1) is unmasked attention."""
    n, d, scale = 23, 6, 0.41
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    ok = True
    for wr, causal in ((0, True), (-1, False)):
        o1, l1 = fwd(q, k, v, scale, -1, wr)
        o2, l2 = A.head_forward(q, k, v, scale, causal)
        ok &= np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12
    return ok


def check_chunked_prefill(fwd):
    """Chunked prefill: the last c rows of square causal attention over N
    tokens equal bottom-right causal attention of those c queries against all
    N keys (the square case needs no alignment convention)."""
    n, c, d, scale = 40, 7, 5, 0.6
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    o_full, l_full = A.head_forward(q, k, v, scale, True)
    o_c, l_c = fwd(q[n - c:], k, v, scale, -1, 0)
    return np.max(np.abs(o_c - o_full[n - c:])) < 1e-12 and np.max(np.abs(l_c - l_full[n - c:])) < 1e-12


def check_window_as_slice(fwd):
    """Row i under the window (wl, wr) equals unmasked attention of query i over
    the slice of keys from position i + off - wl to i + off + wr (clipped to the
    cache), computed with no mask at all."""
    ok = True
    for nq, nk, wl, wr in ((17, 17, 4, 0), (9, 30, 6, 2), (12, 12, 0, 3), (8, 25, 3, -1), (6, 20, -1, 2)):
        d, scale = 4, 0.7
        q, k, v = rnd(nq, d), rnd(nk, d), rnd(nk, d)
        o, lse = fwd(q, k, v, scale, wl, wr)
        for i in range(nq):
            pos = i + nk - nq
            lo = 0 if wl < 0 else max(0, pos - wl)
            hi = nk if wr < 0 else min(nk, pos + wr + 1)
            if hi <= lo:
                ok &= bool(np.all(o[i] == 0)) and lse[i] == -np.inf
                continue
            oi, li = A.head_forward(q[i:i + 1], k[lo:hi], v[lo:hi], scale, False)
            ok &= np.max(np.abs(o[i] - oi[0])) < 1e-12 and abs(lse[i] - li[0]) < 1e-12
    return ok


def check_uniform_window_closed_form(fwd):
    """Q = 0 gives every visible key the same weight: with V_j = j, row i of a
    causal window of w + 1 keys is the mean of max(0, i - w) .. i, and
    lse = ln(count)."""
    n, w = 50, 9
    q, k = np.zeros((n, 3)), rnd(n, 3)
    v = np.arange(n, dtype=np.float64)[:, None]
    o, lse = fwd(q, k, v, 1.3, w, 0)
    lo = np.maximum(0, np.arange(n) - w)
    exp_o = (lo + np.arange(n)) / 2.0
    exp_l = np.log(np.arange(n) - lo + 1)
    return np.max(np.abs(o[:, 0] - exp_o)) < 1e-12 and np.max(np.abs(lse - exp_l)) < 1e-12


def check_brute(fwd, visible_fn):
    """Softmax over the visible scores, against pure-Python loops."""
    nq, nk, d, scale = 6, 11, 4, 0.45
    q, k, v = rnd(nq, d), rnd(nk, d), rnd(nk, d)
    ok = True
    for wl, wr in ((3, 1), (-1, 0), (2, -1), (0, 0)):
        vis = visible_fn(nq, nk, wl, wr)
        o, lse = fwd(q, k, v, scale, wl, wr)
        ob, lb = brute.attention_rows_pred(q.tolist(), k.tolist(), v.tolist(), scale, lambda i, j: bool(vis[i, j]))
        ok &= np.max(np.abs(o - np.array(ob))) < 1e-12
        ok &= bool(np.all((lse == np.array(lb)) | (np.abs(lse - np.array(lb)) < 1e-12)))
    return ok


# ------------------------------------------------------------------ pins

def test_block_mask_golden():
    assert check_block_mask_golden(M.window_visible)


def test_bottom_right_example():
    assert check_bottom_right_example(M.window_visible)


def test_square_causal_matches_square_oracle():
    assert check_square_causal_matches(fwd_with(M.window_visible))


def test_chunked_prefill():
    assert check_chunked_prefill(fwd_with(M.window_visible))


def test_window_equals_attention_over_slice():
    assert check_window_as_slice(fwd_with(M.window_visible))


def test_uniform_window_closed_form():
    assert check_uniform_window_closed_form(fwd_with(M.window_visible))


def test_brute_force():
    assert check_brute(fwd_with(M.window_visible), M.window_visible)


def test_rows_without_keys():
    """Nq > Nk, causal: the first Nq - Nk queries sit before every key."""
    q, k, v = rnd(10, 4), rnd(6, 4), rnd(6, 4)
    o, lse = fwd_with(M.window_visible)(q, k, v, 0.5, -1, 0)
    assert np.all(o[:4] == 0) and np.all(lse[:4] == -np.inf)
    assert np.all(np.isfinite(lse[4:]))


def test_window_wider_than_cache_is_no_bound():
    q, k, v = rnd(9, 4), rnd(21, 4), rnd(21, 4)
    f = fwd_with(M.window_visible)
    o1, l1 = f(q, k, v, 0.5, 21, 0)
    o2, l2 = f(q, k, v, 0.5, -1, 0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _fd_check(nq, nk, hq, hkv, wl, wr, eps=1e-6):
    B, d, scale = 1, 3, 0.8
    q, k, v, do = rnd(B, nq, hq, d), rnd(B, nk, hkv, d), rnd(B, nk, hkv, d), rnd(B, nq, hq, d)
    dq, dk, dv = M.masked_backward(q, k, v, do, scale, wl, wr)

    def loss(q_, k_, v_):
        return float((M.masked_forward(q_, k_, v_, scale, wl, wr)[0] * do).sum())

    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [tuple(RNG.integers(0, s) for s in x.shape) for _ in range(6)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if x is y else y for y in (q, k, v)]
            args_m = [xm if x is y else y for y in (q, k, v)]
            num = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(num - g[idx]) < 1e-6, (idx, num, g[idx])


@pytest.mark.parametrize("nq,nk,hq,hkv,wl,wr", [(5, 9, 2, 1, 3, 1), (7, 7, 2, 2, 2, 0), (4, 12, 3, 1, -1, 0)])
def test_backward_finite_differences(nq, nk, hq, hkv, wl, wr):
    _fd_check(nq, nk, hq, hkv, wl, wr)


def test_unseen_keys_have_zero_gradient():
    """4 queries at the end of 20 keys with a window of 4: keys 0..12 are seen
    by nobody, so their dK and dV vanish exactly."""
    q, k, v, do = rnd(1, 4, 2, 3), rnd(1, 20, 2, 3), rnd(1, 20, 2, 3), rnd(1, 4, 2, 3)
    _, dk, dv = M.masked_backward(q, k, v, do, 0.7, 3, 0)
    assert np.all(dk[:, :13] == 0) and np.all(dv[:, :13] == 0)
    assert np.all(np.abs(dv[:, 13:]).sum(axis=-1) > 0)


def test_varlen_equals_dense_per_sequence():
    lq, lk = [3, 9, 1], [10, 9, 4]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, k, v, do = rnd(sum(lq), 2, 4), rnd(sum(lk), 1, 4), rnd(sum(lk), 1, 4), rnd(sum(lq), 2, 4)
    o, lse = M.masked_varlen_forward(q, k, v, cu_q, cu_k, 0.5, 2, 0)
    dq, dk, dv = M.masked_varlen_backward(q, k, v, do, cu_q, cu_k, 0.5, 2, 0)
    for b in range(3):
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        ob, lb = M.masked_forward(q[None, qs], k[None, ks], v[None, ks], 0.5, 2, 0)
        gb = M.masked_backward(q[None, qs], k[None, ks], v[None, ks], do[None, qs], 0.5, 2, 0)
        assert np.array_equal(o[qs], ob[0]) and np.array_equal(lse[:, qs], lb[0])
        assert np.array_equal(dq[qs], gb[0][0]) and np.array_equal(dk[ks], gb[1][0]) and np.array_equal(dv[ks], gb[2][0])


# ------------------------------------------------------------------ mutation tests
# Plausible mistakes in the visibility matrix; each must fail a pin above.

def mutant_top_left(n_q, n_k, wl, wr):
    pos = np.arange(n_q)[:, None]  # forgot the Nk - Nq shift
    j = np.arange(n_k)[None, :]
    vis = np.ones((n_q, n_k), dtype=bool)
    if wl >= 0:
        vis &= j >= pos - wl
    if wr >= 0:
        vis &= j <= pos + wr
    return vis


def mutant_left_exclusive(n_q, n_k, wl, wr):
    vis = M.window_visible(n_q, n_k, wl, wr)
    if wl >= 0:
        pos = np.arange(n_q)[:, None] + (n_k - n_q)
        vis &= np.arange(n_k)[None, :] > pos - wl
    return vis


def mutant_right_exclusive(n_q, n_k, wl, wr):
    vis = M.window_visible(n_q, n_k, wl, wr)
    if wr >= 0:
        pos = np.arange(n_q)[:, None] + (n_k - n_q)
        vis &= np.arange(n_k)[None, :] < pos + wr
    return vis


def mutant_swapped_sides(n_q, n_k, wl, wr):
    return M.window_visible(n_q, n_k, wr, wl)


def mutant_shift_sign(n_q, n_k, wl, wr):
    pos = np.arange(n_q)[:, None] - (n_k - n_q)
    j = np.arange(n_k)[None, :]
    vis = np.ones((n_q, n_k), dtype=bool)
    if wl >= 0:
        vis &= j >= pos - wl
    if wr >= 0:
        vis &= j <= pos + wr
    return vis


@pytest.mark.parametrize("mutant", [mutant_top_left, mutant_left_exclusive, mutant_right_exclusive,
                                    mutant_swapped_sides, mutant_shift_sign])
def test_visibility_mutants_are_rejected(mutant):
    f = fwd_with(mutant)
    results = [
        check_block_mask_golden(mutant), check_bottom_right_example(mutant), check_square_causal_matches(f),
        check_chunked_prefill(f), check_window_as_slice(f), check_uniform_window_closed_form(f),
    ]
    assert not all(results)


def test_block_mask_golden_rejects_a_wide_window():
    """A window of 200 tokens reaches two tiles back: the golden pattern is
    specific to windows under one tile."""
    vis = M.window_visible(1024, 1024, 199, 0)
    a, b = np.nonzero(M.block_mask(vis, 128))
    assert sorted(set((b - a).tolist())) == [-2, -1, 0]
