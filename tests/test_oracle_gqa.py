"""Pins of the oracle's grouped-query attention."""
import numpy as np
import pytest

from oracle import attention as A
from tests.test_oracle_pins import check_finite_difference

RNG = np.random.default_rng(5)


def rnd(*s):
    return RNG.standard_normal(s)


@pytest.mark.parametrize("causal", [False, True])
def test_group_one_is_plain_attention(causal):
    q, k, v, do = rnd(2, 9, 3, 4), rnd(2, 9, 3, 4), rnd(2, 9, 3, 4), rnd(2, 9, 3, 4)
    o1, l1 = A.gqa_forward(q, k, v, 0.5, causal)
    o2, l2 = A.forward(q, k, v, 0.5, causal)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13
    for g1, g2 in zip(A.gqa_backward(q, k, v, do, 0.5, causal), A.backward(q, k, v, do, 0.5, causal)):
        assert np.max(np.abs(g1 - g2)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_equals_attention_with_repeated_kv(causal):
    """Repeating each K/V head for its group gives ordinary multi-head attention;
    the K/V gradients are the group sums of the repeated heads' gradients."""
    Hq, Hkv = 6, 2
    q, do = rnd(1, 7, Hq, 3), rnd(1, 7, Hq, 3)
    k, v = rnd(1, 7, Hkv, 3), rnd(1, 7, Hkv, 3)
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    o1, l1 = A.gqa_forward(q, k, v, 0.7, causal)
    o2, l2 = A.forward(q, kr, vr, 0.7, causal)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13
    dq1, dk1, dv1 = A.gqa_backward(q, k, v, do, 0.7, causal)
    dq2, dk2, dv2 = A.backward(q, kr, vr, do, 0.7, causal)
    assert np.max(np.abs(dq1 - dq2)) < 1e-12
    assert np.max(np.abs(dk1 - dk2.reshape(1, 7, Hkv, Hq // Hkv, 3).sum(3))) < 1e-12
    assert np.max(np.abs(dv1 - dv2.reshape(1, 7, Hkv, Hq // Hkv, 3).sum(3))) < 1e-12


def test_gqa_backward_finite_difference():
    """Central differences of sum(dO * O) over the shared K/V of a 2-query-head group."""
    Hq, Hkv, n, d = 2, 1, 6, 3
    q, k, v, do = rnd(1, n, Hq, d), rnd(1, n, Hkv, d), rnd(1, n, Hkv, d), rnd(1, n, Hq, d)
    grads = A.gqa_backward(q, k, v, do, 0.6, True)

    def loss(qq, kk, vv):
        return float(np.sum(do * A.gqa_forward(qq, kk, vv, 0.6, True)[0]))

    h = 1e-6
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (lp - loss(*args)) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(num) < 1e-6


def test_gqa_decode_equals_repeated():
    q = rnd(2, 1, 8, 4)
    kc, vc = rnd(2, 11, 2, 4), rnd(2, 11, 2, 4)
    o1, l1 = A.gqa_decode_forward(q, kc, vc, 0.5)
    o2, l2 = A.decode_forward(q, np.repeat(kc, 4, axis=2), np.repeat(vc, 4, axis=2), 0.5)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13
