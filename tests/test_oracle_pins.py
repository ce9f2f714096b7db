"""Pins of the float64 oracle against facts that do not come from the oracle.

Each check is written as a function of the implementation under test so that
the mutation tests at the bottom can plant a plausible mistake in a copy of the
oracle (on the CPU) and show that at least one pin rejects it.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def rnd(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ------------------------------------------------------------------ checks

def check_brute(head_fwd, causal, n=9, d=5, scale=0.37):
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    o, lse = head_fwd(q, k, v, scale, causal)
    ob, lb = brute.attention_rows(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    return np.max(np.abs(o - np.array(ob))) < 1e-12 and np.max(np.abs(lse - np.array(lb))) < 1e-12


def check_shift(head_fwd, causal, c=1000.0):
    """Add a per-row constant to every score through an extra coordinate:
    q' = [q, c_i], k' = [k, 1] gives S'_ij = S_ij + scale*c_i.  O must not
    change and lse must move by scale*c_i (softmax(x - c) = softmax(x))."""
    n, d, scale = 12, 6, 0.5
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    ci = c * (1.0 + RNG.random(n))
    q2 = np.concatenate([q, ci[:, None]], 1)
    k2 = np.concatenate([k, np.ones((n, 1))], 1)
    o1, l1 = head_fwd(q, k, v, scale, causal)
    o2, l2 = head_fwd(q2, k2, v, scale, causal)
    if not (np.all(np.isfinite(o2)) and np.all(np.isfinite(l2))):
        return False
    return np.max(np.abs(o1 - o2)) < 1e-9 and np.max(np.abs(l2 - l1 - scale * ci)) < 1e-9


def check_uniform_closed_form(head_fwd, causal, n=11, d=4):
    """Q = 0: every visible key gets the same weight.  Non-causal O_i = mean(V),
    lse_i = ln N; causal O_i = mean(V_0..V_i), lse_i = ln(i+1)."""
    q, k, v = np.zeros((n, d)), rnd(n, d), rnd(n, d)
    o, lse = head_fwd(q, k, v, 0.9, causal)
    if causal:
        exp_o = np.cumsum(v, 0) / np.arange(1, n + 1)[:, None]
        exp_l = np.log(np.arange(1, n + 1))
    else:
        exp_o = np.tile(v.mean(0), (n, 1))
        exp_l = np.full(n, math.log(n))
    return np.max(np.abs(o - exp_o)) < 1e-12 and np.max(np.abs(lse - exp_l)) < 1e-12


def check_causal_first_row(head_fwd, n=10, d=7, scale=0.3):
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    o, lse = head_fwd(q, k, v, scale, True)
    return np.max(np.abs(o[0] - v[0])) < 1e-13 and abs(lse[0] - scale * q[0] @ k[0]) < 1e-12


def check_causal_last_row(head_fwd, n=10, d=7, scale=0.3):
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    oc, lc = head_fwd(q, k, v, scale, True)
    on, ln = head_fwd(q, k, v, scale, False)
    return np.max(np.abs(oc[-1] - on[-1])) < 1e-13 and abs(lc[-1] - ln[-1]) < 1e-12


def check_constant_v(head_fwd, causal):
    n, d = 9, 5
    q, k = rnd(n, d, scale=3), rnd(n, d, scale=3)
    row = rnd(d)
    v = np.tile(row, (n, 1))
    o, _ = head_fwd(q, k, v, 0.7, causal)
    return np.max(np.abs(o - row)) < 1e-12


def check_one_hot(head_fwd):
    """A key aligned with the query and scaled far above the rest takes all
    the weight: O_i -> V_j."""
    n, d = 8, 8
    k, _ = np.linalg.qr(rnd(n, d))   # orthonormal keys: q.k = 60 for the match, 0 otherwise
    v = rnd(n, d)
    q = 60.0 * k[[3, 5, 0, 7, 1, 2, 6, 4]]
    o, _ = head_fwd(q, k, v, 1.0, False)
    return np.max(np.abs(o - v[[3, 5, 0, 7, 1, 2, 6, 4]])) < 1e-6


def check_permutation(head_fwd):
    n, d = 10, 4
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    perm = RNG.permutation(n)
    o1, l1 = head_fwd(q, k, v, 0.5, False)
    o2, l2 = head_fwd(q, k[perm], v[perm], 0.5, False)
    return np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def check_scale(head_fwd, causal):
    n, d = 7, 3
    q, k, v = rnd(n, d), rnd(n, d), rnd(n, d)
    o1, l1 = head_fwd(q, k, v, 0.25, causal)
    o2, l2 = head_fwd(0.25 * q, k, v, 1.0, causal)
    return np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def check_finite_difference(head_bwd, head_fwd, causal, n=8, d=4, scale=0.6, h=1e-6):
    """Central differences of L = sum(dO * O) against the analytic gradients."""
    q, k, v, do = rnd(n, d), rnd(n, d), rnd(n, d), rnd(n, d)
    grads = head_bwd(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _ = head_fwd(qq, kk, vv, scale, causal)
        return float(np.sum(do * o))

    worst = 0.0
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            num[idx] = (lp - lm) / (2 * h)
        worst = max(worst, np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-30))
    return worst < 1e-6


def check_merge(partials, merge, dense, num_splits):
    B, H, L, d = 2, 3, 37, 5
    q = rnd(B, 1, H, d)
    kc, vc = rnd(B, L, H, d, scale=2.0), rnd(B, L, H, d)
    o_ref, l_ref = dense(q, kc, vc, 0.4)
    op, lp = partials(q, kc, vc, 0.4, num_splits)
    o, l = merge(op, lp)
    return np.max(np.abs(o - o_ref[:, 0])) < 1e-12 and np.max(np.abs(l - l_ref)) < 1e-12


def check_varlen(varlen_fwd, head_fwd, causal):
    lengths = [5, 1, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    total, H, d = int(cu[-1]), 2, 4
    q, k, v = rnd(total, H, d), rnd(total, H, d), rnd(total, H, d)
    o, lse = varlen_fwd(q, k, v, cu, 0.5, causal)
    for b in range(len(lengths)):
        lo, hi = cu[b], cu[b + 1]
        for h in range(H):
            oh, lh = head_fwd(q[lo:hi, h], k[lo:hi, h], v[lo:hi, h], 0.5, causal)
            if np.max(np.abs(o[lo:hi, h] - oh)) > 1e-13 or np.max(np.abs(lse[h, lo:hi] - lh)) > 1e-13:
                return False
    return True


# ------------------------------------------------------------------ pins of the oracle

@pytest.mark.parametrize("causal", [False, True])
def test_brute_force(causal):
    assert check_brute(A.head_forward, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    p = A.head_probs(rnd(13, 6), rnd(13, 6), 0.8, causal)
    assert np.all(p >= 0)
    assert np.max(np.abs(p.sum(1) - 1)) < 1e-12
    if causal:
        assert np.all(np.triu(p, 1) == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariance(causal):
    assert check_shift(A.head_forward, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_closed_form(causal):
    assert check_uniform_closed_form(A.head_forward, causal)


def test_causal_first_row_closed_form():
    assert check_causal_first_row(A.head_forward)


def test_causal_last_row_is_unmasked():
    assert check_causal_last_row(A.head_forward)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_rows(causal):
    assert check_constant_v(A.head_forward, causal)


def test_one_hot():
    assert check_one_hot(A.head_forward)


def test_key_permutation():
    assert check_permutation(A.head_forward)


@pytest.mark.parametrize("causal", [False, True])
def test_scale_folds_into_q(causal):
    assert check_scale(A.head_forward, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_difference(causal):
    assert check_finite_difference(A.head_backward, A.head_forward, causal)


def test_backward_uniform_closed_form():
    """Q = 0 (non-causal): P = 1/N, so dV_j = mean_i dO_i for every j."""
    n, d = 9, 4
    q, k, v, do = np.zeros((n, d)), rnd(n, d), rnd(n, d), rnd(n, d)
    _, _, dv = A.head_backward(q, k, v, do, 0.5, False)
    assert np.max(np.abs(dv - do.mean(0))) < 1e-12


def test_backward_constant_v_gives_zero_qk_grads():
    """With equal V rows, O does not depend on Q or K."""
    n, d = 9, 4
    v = np.tile(rnd(d), (n, 1))
    dq, dk, _ = A.head_backward(rnd(n, d), rnd(n, d), v, rnd(n, d), 0.5, True)
    assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12


def test_dense_batch_matches_heads():
    B, N, H, d = 2, 6, 3, 4
    q, k, v, do = rnd(B, N, H, d), rnd(B, N, H, d), rnd(B, N, H, d), rnd(B, N, H, d)
    o, lse = A.forward(q, k, v, 0.5, True)
    dq, dk, dv = A.backward(q, k, v, do, 0.5, True)
    for b in range(B):
        for h in range(H):
            oh, lh = brute.attention_rows(q[b, :, h].tolist(), k[b, :, h].tolist(), v[b, :, h].tolist(), 0.5, True)
            assert np.max(np.abs(o[b, :, h] - np.array(oh))) < 1e-12
            assert np.max(np.abs(lse[b, h] - np.array(lh))) < 1e-12
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_per_sequence(causal):
    assert check_varlen(A.varlen_forward, A.head_forward, causal)


def test_varlen_backward_equals_per_sequence():
    lengths = [4, 7]
    cu = [0, 4, 11]
    q, k, v, do = rnd(11, 2, 3), rnd(11, 2, 3), rnd(11, 2, 3), rnd(11, 2, 3)
    dq, dk, dv = A.varlen_backward(q, k, v, do, cu, 0.5, True)
    for b in range(2):
        lo, hi = cu[b], cu[b + 1]
        for h in range(2):
            g = A.head_backward(q[lo:hi, h], k[lo:hi, h], v[lo:hi, h], do[lo:hi, h], 0.5, True)
            for got, want in zip((dq, dk, dv), g):
                assert np.max(np.abs(got[lo:hi, h] - want)) < 1e-13


@pytest.mark.parametrize("num_splits", [1, 2, 3, 8, 40])
def test_split_merge_equals_dense(num_splits):
    assert check_merge(A.decode_partials, A.merge_partials, A.decode_forward, num_splits)


@pytest.mark.parametrize("block_c", [1, 7, 64, 1000])
@pytest.mark.parametrize("tau", [0.0, 8.0, 30.0])
@pytest.mark.parametrize("causal", [False, True])
def test_online_equals_batch(block_c, tau, causal):
    n, d = 67, 8
    q, k, v = rnd(n, d, scale=2.0), rnd(n, d, scale=2.0), rnd(n, d)
    o, lse, _ = A.online_head_forward(q, k, v, 0.6, causal, block_c, tau)
    o_ref, l_ref = A.head_forward(q, k, v, 0.6, causal)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - l_ref)) < 1e-12


def test_lazy_rescale_takes_fewer_rescales():
    """Raising the threshold skips rescales without changing the result."""
    n, d = 512, 16
    q, k, v = rnd(n, d, scale=1.5), rnd(n, d, scale=1.5), rnd(n, d)
    counts = [A.online_head_forward(q, k, v, 1.0, True, 16, tau)[2] for tau in (0.0, 8.0, 1e9)]
    assert counts[0] > counts[1] > counts[2] == 0


def test_top_left_causal_golden():
    g = json.load(open(os.path.join(GOLDEN, "pages_worked_numbers.json")))["top_left_causal"]
    nq, nk = g["n_q"], g["n_k"]
    q, k = rnd(nq, 4), rnd(nk, 4)
    v = np.eye(nk)[:, :nk]  # O row = the attention weights themselves
    o_tl, _ = A.head_forward(q, k, v, 1.0, True, q_pos=np.arange(nq))
    assert list(np.nonzero(o_tl[0] > 0)[0]) == g["first_query_visible_keys_top_left"]
    # the library's convention (bottom-right) lets the first of 4 queries see keys 0..124
    o_br, _ = A.head_forward(q, k, v, 1.0, True)
    assert np.count_nonzero(o_br[0] > 0) == nk - nq + 1


# ------------------------------------------------------------------ mutation tests
# Each mutant is a copy of an oracle function with one plausible mistake,
# several of them the broken exercise stubs printed on the pages.  At least
# one pin must reject every mutant.

def mutant_no_max_subtraction(q, k, v, scale, causal, q_pos=None):
    # the "partial_attention" stub: exponentiate raw scores
    s = scale * (np.asarray(q) @ np.asarray(k).T)
    if causal:
        s = np.where(np.arange(len(k))[None, :] <= np.arange(len(q))[:, None], s, -np.inf)
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(s)
        l = e.sum(1)
        return (e / l[:, None]) @ v, np.log(l)


def mutant_mask_off_by_one(q, k, v, scale, causal, q_pos=None):
    n = len(q)
    pos = np.arange(n) - 1 if causal else None
    if causal:
        s = scale * (q @ k.T)
        s = np.where(np.arange(len(k))[None, :] <= pos[:, None], s, -np.inf)
        s[0, 0] = scale * q[0] @ k[0]
        m = s.max(1)
        e = np.exp(s - m[:, None])
        return (e / e.sum(1)[:, None]) @ v, m + np.log(e.sum(1))
    return A.head_forward(q, k, v, scale, causal)


def mutant_transposed_mask(q, k, v, scale, causal, q_pos=None):
    s = scale * (q @ k.T)
    if causal:
        s = np.where(np.arange(len(k))[None, :] >= np.arange(len(q))[:, None], s, -np.inf)
    m = s.max(1)
    e = np.exp(s - m[:, None])
    return (e / e.sum(1)[:, None]) @ v, m + np.log(e.sum(1))


def mutant_lse_log2(q, k, v, scale, causal, q_pos=None):
    o, lse = A.head_forward(q, k, v, scale, causal)
    return o, lse / math.log(2.0)


def mutant_missing_scale_in_lse(q, k, v, scale, causal, q_pos=None):
    o, _ = A.head_forward(q, k, v, scale, causal)
    _, lse1 = A.head_forward(q, k, v, 1.0, causal)
    return o, lse1


@pytest.mark.parametrize("mutant", [mutant_no_max_subtraction, mutant_mask_off_by_one,
                                    mutant_transposed_mask, mutant_lse_log2,
                                    mutant_missing_scale_in_lse])
def test_forward_mutants_are_rejected(mutant):
    results = [
        check_brute(mutant, False), check_brute(mutant, True),
        check_shift(mutant, False), check_shift(mutant, True),
        check_uniform_closed_form(mutant, True), check_causal_first_row(mutant),
        check_scale(mutant, True),
    ]
    assert not all(results)


def mutant_bwd_missing_dsum(q, k, v, do, scale, causal):
    p = A.head_probs(q, k, scale, causal)
    dp = do @ v.T
    ds = p * dp
    return scale * ds @ k, scale * ds.T @ q, p.T @ do


def mutant_bwd_missing_scale(q, k, v, do, scale, causal):
    dq, dk, dv = A.head_backward(q, k, v, do, scale, causal)
    return dq / scale, dk / scale, dv


def mutant_bwd_transposed_dv(q, k, v, do, scale, causal):
    dq, dk, _ = A.head_backward(q, k, v, do, scale, causal)
    p = A.head_probs(q, k, scale, causal)
    return dq, dk, p @ do


@pytest.mark.parametrize("mutant", [mutant_bwd_missing_dsum, mutant_bwd_missing_scale,
                                    mutant_bwd_transposed_dv])
def test_backward_mutants_are_rejected(mutant):
    assert not (check_finite_difference(mutant, A.head_forward, False)
                and check_finite_difference(mutant, A.head_forward, True))


def mutant_equal_weight_merge(o_parts, lse_parts):
    # the "combine" stub: equal weights and the max of the lses
    return np.mean(o_parts, axis=-2), np.max(lse_parts, axis=-1)


def test_equal_weight_merge_is_rejected():
    assert not check_merge(A.decode_partials, mutant_equal_weight_merge, A.decode_forward, 4)


def mutant_varlen_across_sequences(q, k, v, cu, scale, causal):
    # the "varlen_attention" stub: one attention over all packed rows
    total, H, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((H, total))
    for h in range(H):
        o[:, h], lse[h] = A.head_forward(q[:, h], k[:, h], v[:, h], scale, causal)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_across_sequences_is_rejected(causal):
    assert not check_varlen(mutant_varlen_across_sequences, A.head_forward, causal)
