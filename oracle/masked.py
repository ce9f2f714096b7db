"""Float64 CPU oracle for masked attention: causal and sliding-window masks with
their own query and key lengths.

TEST INFRASTRUCTURE ONLY, like ``oracle.attention``: imported by ``tests/``
and never by the library.

What it computes is the dense definition: build the boolean visibility matrix,
set the hidden scores to -inf, take the softmax of each row, multiply by V.

Sources (zerotofrontier.app "efficient-attention/flash-2-3", section "Using
it, the real way"):
  * FlashAttention kernels handle causal masks, sliding windows and variable
    lengths themselves;
  * PyTorch's ``is_causal`` aligns the mask to the top left, which is wrong for
    chunked prefill or decoding against a cache; the flash-attn package's
    ``causal=True`` aligns it to the bottom right;
  * FlexAttention's block mask marks the 128 x 128 tiles that hold no visible
    score so the kernel can skip them; with a 64-token window only the
    diagonal tiles and the ones just below them remain.

Reading (the pages name the conventions but print no formula): query i of a
sequence with Nq queries and Nk keys sits at key position i + Nk - Nq
(bottom-right), and a window (window_left, window_right) lets it see the keys

    i + Nk - Nq - window_left  <=  j  <=  i + Nk - Nq + window_right,

with -1 leaving a side open: (-1, -1) is no mask, (-1, 0) causal, (w, 0) a
causal sliding window of w + 1 keys.  A row that sees no key has O = 0 and
lse = -inf, as in ``oracle.attention``.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

NEG_INF = -np.inf


def window_visible(n_q: int, n_k: int, window_left: int, window_right: int) -> np.ndarray:
    """Boolean [n_q, n_k]: entry (i, j) is True when query i sees key j."""
    pos = np.arange(n_q)[:, None] + (n_k - n_q)  # each query's key position
    j = np.arange(n_k)[None, :]
    vis = np.ones((n_q, n_k), dtype=bool)
    if window_left >= 0:
        vis &= j >= pos - window_left
    if window_right >= 0:
        vis &= j <= pos + window_right
    return vis


def top_left_causal_visible(n_q: int, n_k: int) -> np.ndarray:
    """PyTorch's ``is_causal`` convention, for contrast: query i sees keys 0..i."""
    return np.arange(n_k)[None, :] <= np.arange(n_q)[:, None]


def block_mask(visible: np.ndarray, tile: int = 128) -> np.ndarray:
    """Tiles [n_q / tile, n_k / tile] (rounded up) that hold at least one
    visible score: the tiles a block-sparse kernel has to visit."""
    n_q, n_k = visible.shape
    tq, tk = -(-n_q // tile), -(-n_k // tile)
    out = np.zeros((tq, tk), dtype=bool)
    for a in range(tq):
        for b in range(tk):
            out[a, b] = visible[a * tile:(a + 1) * tile, b * tile:(b + 1) * tile].any()
    return out


def head_forward_visible(q, k, v, scale: float, visible: np.ndarray):
    """One head under an explicit visibility matrix.  q [Nq, d], k/v [Nk, d]
    float64 -> (o [Nq, d], lse [Nq])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = np.where(visible, scale * (q @ k.T), NEG_INF)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], NEG_INF)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l[:, None] > 0, e / l[:, None], 0.0)
        lse = np.where(l > 0, m_safe + np.log(l), NEG_INF)
    return p @ v, lse


def head_backward_visible(q, k, v, do, scale: float, visible: np.ndarray):
    """Gradients of sum(dO * O) for one head under a visibility matrix:
    dV = P^T dO, dP = dO V^T, D = rowsum(P * dP), dS = P (dP - D),
    dQ = scale dS K, dK = scale dS^T Q."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    s = np.where(visible, scale * (q @ k.T), NEG_INF)
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l[:, None] > 0, e / l[:, None], 0.0)
    dv = p.T @ do
    dp = do @ v.T
    dsum = (p * dp).sum(axis=1)
    ds = p * (dp - dsum[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv


def masked_forward(q, k, v, scale: float, window_left: int, window_right: int):
    """Dense batch: q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d] (Hkv divides Hq; query
    head h reads K/V head h // (Hq / Hkv)) -> (o [B, Nq, Hq, d], lse [B, Hq, Nq])."""
    B, n_q, Hq, _ = q.shape
    n_k, Hkv = k.shape[1], k.shape[2]
    group = Hq // Hkv
    vis = window_visible(n_q, n_k, window_left, window_right)
    o = np.zeros((B, n_q, Hq, v.shape[-1]))
    lse = np.zeros((B, Hq, n_q))
    for b in range(B):
        for h in range(Hq):
            oh, lh = head_forward_visible(q[b, :, h], k[b, :, h // group], v[b, :, h // group], scale, vis)
            o[b, :, h] = oh
            lse[b, h] = lh
    return o, lse


def masked_backward(q, k, v, do, scale: float, window_left: int, window_right: int):
    """Gradients of masked_forward; dK and dV of a K/V head sum over its query heads."""
    B, n_q, Hq, _ = q.shape
    n_k, Hkv = k.shape[1], k.shape[2]
    group = Hq // Hkv
    vis = window_visible(n_q, n_k, window_left, window_right)
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            g = head_backward_visible(q[b, :, h], k[b, :, h // group], v[b, :, h // group], do[b, :, h], scale, vis)
            dq[b, :, h] = g[0]
            dk[b, :, h // group] += g[1]
            dv[b, :, h // group] += g[2]
    return dq, dk, dv


def masked_varlen_forward(q, k, v, cu_q: Sequence[int], cu_k: Sequence[int], scale: float, window_left: int,
                          window_right: int):
    """Packed batch: sequence b owns query rows cu_q[b]..cu_q[b+1]-1 and key rows
    cu_k[b]..cu_k[b+1]-1; the mask aligns them at the bottom right.
    q [total_q, Hq, d], k/v [total_k, Hkv, d] -> (o [total_q, Hq, d], lse [Hq, total_q])."""
    Hq = q.shape[1]
    group = Hq // k.shape[1]
    o = np.zeros((q.shape[0], Hq, v.shape[-1]))
    lse = np.zeros((Hq, q.shape[0]))
    for b in range(len(cu_q) - 1):
        qa, qb, ka, kb = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        vis = window_visible(qb - qa, kb - ka, window_left, window_right)
        for h in range(Hq):
            oh, lh = head_forward_visible(q[qa:qb, h], k[ka:kb, h // group], v[ka:kb, h // group], scale, vis)
            o[qa:qb, h] = oh
            lse[h, qa:qb] = lh
    return o, lse


def masked_varlen_backward(q, k, v, do, cu_q: Sequence[int], cu_k: Sequence[int], scale: float, window_left: int,
                           window_right: int):
    """Gradients of masked_varlen_forward."""
    Hq = q.shape[1]
    group = Hq // k.shape[1]
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(len(cu_q) - 1):
        qa, qb, ka, kb = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        vis = window_visible(qb - qa, kb - ka, window_left, window_right)
        for h in range(Hq):
            g = head_backward_visible(q[qa:qb, h], k[ka:kb, h // group], v[ka:kb, h // group], do[qa:qb, h],
                                      scale, vis)
            dq[qa:qb, h] = g[0]
            dk[ka:kb, h // group] += g[1]
            dv[ka:kb, h // group] += g[2]
    return dq, dk, dv
