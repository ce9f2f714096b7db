"""Plain float64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it and shares no code with it.

What it computes is the plain definition of attention, materialising the score
matrix S and the probability matrix P for one (batch, head) at a time:

    S = scale * Q K^T                       (causal: S_ij = -inf where key j lies
                                             after query i)
    m_i = max_j S_ij
    P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)
    O = P V
    lse_i = m_i + ln sum_j exp(S_ij - m_i)   (natural log, scale included)

Sources: "13.14 FlashAttention: IO-aware exact attention" (textbookofai.com),
sections "Memory bandwidth as the bottleneck" (S = QK^T, softmax, P V) and
"Online softmax" (subtracting the running maximum before exponentiating; the
tiled result is exact); "Flash Attention and the Online-Softmax Trick"
(s-samarth.github.io) section 1 (S = QK^T -> P = softmax(S) -> O = PV) and
section 3 (softmax(x - c) = softmax(x)).  The log-sum-exp ``lse = m + log l`` is
the quantity that FlashAttention-2 keeps for the backward pass
(zerotofrontier.app "efficient-attention/flash-2-3", section "Fewer non-matmul
FLOPs").

The backward pass is the standard derivative of softmax attention (the pages
only say that the backward recomputes P from lse, same section):

    dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P * (dP - D),
    dQ = scale * dS K,  dK = scale * dS^T Q.

Causal alignment: key j is visible to query i iff j <= i + (Nk - Nq), i.e. the
bottom-right convention of the flash-attn package ("Using it, the real way").
It equals PyTorch's top-left convention whenever Nq == Nk, which is every
causal case of this library.

A row whose keys are all masked has O = 0 and lse = -inf (the pages are silent;
this is the convention the kernels follow too).

Layouts follow the flash-attn calls the pages print: dense [B, N, H, d],
packed variable length [total, H, d] with int32 ``cu_seqlens`` of length B+1
(section "Variable-length batches without padding"), lse [B, H, N] dense and
[H, total] packed.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

NEG_INF = -np.inf


def _causal_visible(q_pos: np.ndarray, n_k: int) -> np.ndarray:
    """Boolean [len(q_pos), n_k]: key j is visible to the query at position q_pos[i]
    iff j <= q_pos[i]."""
    j = np.arange(n_k)[None, :]
    return j <= np.asarray(q_pos)[:, None]


def _default_pos(n_q: int, n_k: int) -> np.ndarray:
    # bottom-right alignment: the last query sits at the last key
    return np.arange(n_q) + (n_k - n_q)


def _scores(q, k, scale, causal, q_pos):
    s = scale * (q @ k.T)
    if causal:
        s = np.where(_causal_visible(q_pos, k.shape[0]), s, NEG_INF)
    return s


def head_forward(q, k, v, scale: float, causal: bool, q_pos: Optional[np.ndarray] = None):
    """One head.  q [Nq, d], k/v [Nk, d] float64 -> (o [Nq, d], lse [Nq]).

    ``q_pos`` gives each query row's position among the keys (default: the
    bottom-right alignment, 0..Nq-1 when Nq == Nk) so that a sample of rows
    can be evaluated on its own."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if q_pos is None:
        q_pos = _default_pos(q.shape[0], k.shape[0])
    s = _scores(q, k, scale, causal, q_pos)
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l[:, None] > 0, e / l[:, None], 0.0)
        lse = np.where(l > 0, m_safe + np.log(l), NEG_INF)
    o = p @ v
    return o, lse


def head_probs(q, k, scale: float, causal: bool):
    """P for one head (used by the invariance pins and the backward pass)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    s = _scores(q, k, scale, causal, _default_pos(q.shape[0], k.shape[0]))
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(l[:, None] > 0, e / l[:, None], 0.0)


def head_backward(q, k, v, do, scale: float, causal: bool):
    """One head: gradients of sum(dO * O) with respect to q, k, v."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    p = head_probs(q, k, scale, causal)
    dv = p.T @ do
    dp = do @ v.T
    dsum = (p * dp).sum(axis=1)
    ds = p * (dp - dsum[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


# ---------------------------------------------------------------- dense [B, N, H, d]

def forward(q, k, v, scale: float, causal: bool):
    """Dense batch: q, k, v [B, N, H, d] -> (o [B, N, H, d], lse [B, H, N])."""
    B, N, H, d = q.shape
    o = np.zeros((B, N, H, v.shape[-1]))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            oh, lh = head_forward(q[b, :, h], k[b, :, h], v[b, :, h], scale, causal)
            o[b, :, h] = oh
            lse[b, h] = lh
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool):
    """Dense batch gradients, each [B, N, H, d]."""
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    B, N, H, d = q.shape
    for b in range(B):
        for h in range(H):
            gq, gk, gv = head_backward(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], scale, causal)
            dq[b, :, h], dk[b, :, h], dv[b, :, h] = gq, gk, gv
    return dq, dk, dv


# ---------------------------------------------------------------- packed variable length

def varlen_forward(q, k, v, cu_seqlens: Sequence[int], scale: float, causal: bool):
    """Packed batch: q, k, v [total, H, d]; sequence b owns rows
    cu_seqlens[b] .. cu_seqlens[b+1]-1 and attends only inside them
    (block-diagonal document mask).  Returns o [total, H, d], lse [H, total]."""
    cu = [int(x) for x in cu_seqlens]
    total, H, d = q.shape
    o = np.zeros((total, H, v.shape[-1]))
    lse = np.zeros((H, total))
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        if hi <= lo:
            continue
        for h in range(H):
            oh, lh = head_forward(q[lo:hi, h], k[lo:hi, h], v[lo:hi, h], scale, causal)
            o[lo:hi, h] = oh
            lse[h, lo:hi] = lh
    return o, lse


def varlen_backward(q, k, v, do, cu_seqlens: Sequence[int], scale: float, causal: bool):
    cu = [int(x) for x in cu_seqlens]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    H = q.shape[1]
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        if hi <= lo:
            continue
        for h in range(H):
            gq, gk, gv = head_backward(q[lo:hi, h], k[lo:hi, h], v[lo:hi, h], do[lo:hi, h], scale, causal)
            dq[lo:hi, h], dk[lo:hi, h], dv[lo:hi, h] = gq, gk, gv
    return dq, dk, dv


# ---------------------------------------------------------------- single-token decode

def decode_forward(q, k_cache, v_cache, scale: float):
    """One new query per sequence against its whole cache, no mask.
    q [B, 1, H, d], caches [B, L, H, d] -> (o [B, 1, H, d], lse [B, H])."""
    B, _, H, d = q.shape
    o = np.zeros((B, 1, H, v_cache.shape[-1]))
    lse = np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            oh, lh = head_forward(q[b, :, h], k_cache[b, :, h], v_cache[b, :, h], scale, False)
            o[b, 0, h] = oh[0]
            lse[b, h] = lh[0]
    return o, lse


def split_bounds(L: int, num_splits: int):
    """Chunk c of a length-L cache covers keys [c*ceil(L/S), min(L, (c+1)*ceil(L/S)))."""
    chunk = -(-L // num_splits)
    return [(c * chunk, min(L, (c + 1) * chunk)) for c in range(num_splits)]


def decode_partials(q, k_cache, v_cache, scale: float, num_splits: int):
    """Flash-Decoding split step ("Decoding needs a different split"): each chunk
    of the cache reports its own normalised output and its log-sum-exp.
    Returns o_parts [B, H, S, d], lse_parts [B, H, S] (an empty chunk has
    O = 0 and lse = -inf)."""
    B, _, H, d = q.shape
    L = k_cache.shape[1]
    bounds = split_bounds(L, num_splits)
    o_parts = np.zeros((B, H, num_splits, v_cache.shape[-1]))
    lse_parts = np.full((B, H, num_splits), NEG_INF)
    for b in range(B):
        for h in range(H):
            for c, (lo, hi) in enumerate(bounds):
                if hi <= lo:
                    continue
                oc, lc = head_forward(q[b, :, h], k_cache[b, lo:hi, h], v_cache[b, lo:hi, h], scale, False)
                o_parts[b, h, c] = oc[0]
                lse_parts[b, h, c] = lc[0]
    return o_parts, lse_parts


def merge_partials(o_parts, lse_parts):
    """Flash-Decoding merge: the output is the average of the chunks' outputs
    weighted by their softmax mass, lse = ln sum_c exp(lse_c) and
    O = sum_c exp(lse_c - lse) O_c (the displayed formula after the chunking
    paragraph did not survive extraction; this is the log-sum-exp merge its
    prose describes).  Inputs [..., S, d] and [..., S]."""
    lse_parts = np.asarray(lse_parts, np.float64)
    m = lse_parts.max(axis=-1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe[..., None])
    total = w.sum(axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(total > 0, m_safe + np.log(total), NEG_INF)
        wn = np.where(total[..., None] > 0, w / total[..., None], 0.0)
    o = (wn[..., None] * np.asarray(o_parts, np.float64)).sum(axis=-2)
    return o, lse


# ---------------------------------------------------------------- the tiled algorithm

def online_head_forward(q, k, v, scale: float, causal: bool, block_c: int, tau_log2: float = 0.0):
    """The one-pass tiled algorithm, in float64, in the pages' order.

    For each block of ``block_c`` keys: take the block's row maximum, update the
    running maximum, rescale the running denominator l and the unnormalised
    output O~ by exp(m_old - m_new), add the block's exponentials and their
    product with V, and divide by l once at the end ("Online softmax";
    FlashAttention-2 "Fewer non-matmul FLOPs").

    ``tau_log2`` is the conditional-rescaling threshold of the Blackwell
    design ("And on Blackwell"): the reference point m_ref moves to the new
    maximum only when the maximum has grown by more than tau (in log2 units,
    i.e. by more than a factor 2**tau); otherwise the stale m_ref stays and the
    block's exponentials may exceed 1 by up to 2**tau.  tau = 0 is the classic
    algorithm.  Any reference point gives the same result because l and O~
    share it.  Returns (o, lse, number_of_rescales)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n_q, n_k = q.shape[0], k.shape[0]
    tau = tau_log2 * math.log(2.0)
    m_ref = np.full(n_q, NEG_INF)
    l = np.zeros(n_q)
    o_acc = np.zeros((n_q, v.shape[1]))
    rescales = 0
    rows = np.arange(n_q)
    for j0 in range(0, n_k, block_c):
        j1 = min(n_k, j0 + block_c)
        s = scale * (q @ k[j0:j1].T)
        if causal:
            s = np.where(np.arange(j0, j1)[None, :] <= rows[:, None], s, NEG_INF)
        m_blk = s.max(axis=1)
        grow = m_blk > m_ref + tau
        # rows whose reference point moves: rescale l and O~ by exp(m_old - m_new)
        with np.errstate(invalid="ignore"):
            alpha = np.where(grow, np.exp(np.where(np.isfinite(m_ref), m_ref - m_blk, NEG_INF)), 1.0)
        rescales += int(np.sum(grow & np.isfinite(m_ref)))
        m_ref = np.where(grow, m_blk, m_ref)
        l = l * alpha
        o_acc = o_acc * alpha[:, None]
        m_use = np.where(np.isfinite(m_ref), m_ref, 0.0)
        p = np.exp(s - m_use[:, None])
        l = l + p.sum(axis=1)
        o_acc = o_acc + p @ v[j0:j1]
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(l[:, None] > 0, o_acc / l[:, None], 0.0)
        lse = np.where(l > 0, np.where(np.isfinite(m_ref), m_ref, 0.0) + np.log(l), NEG_INF)
    return o, lse, rescales


# ---------------------------------------------------------------- paged KV cache

def gather_pages(pages, block_table_row, seq_len: int):
    """One sequence's cache from a page pool ("Paged KV caches, a preview of
    serving"): logical block j of page_size keys lives in physical page
    block_table_row[j]; only the first seq_len keys belong to the sequence (the
    rest of its last page are unused slots).  pages [num_pages, P, H, d]."""
    P = pages.shape[1]
    n_blocks = -(-seq_len // P)
    rows = [pages[int(block_table_row[j])] for j in range(n_blocks)]
    if not rows:
        return np.zeros((0,) + pages.shape[2:])
    return np.concatenate(rows, axis=0)[:seq_len]


def paged_decode_forward(q, k_pages, v_pages, block_table, seq_lens, scale: float):
    """Decode against paged caches: each sequence attends to exactly its own
    seq_len keys.  q [B, 1, H, d] -> (o [B, 1, H, d], lse [B, H])."""
    B, _, H, d = q.shape
    o = np.zeros((B, 1, H, v_pages.shape[-1]))
    lse = np.zeros((B, H))
    for b in range(B):
        kb = gather_pages(k_pages, block_table[b], int(seq_lens[b]))
        vb = gather_pages(v_pages, block_table[b], int(seq_lens[b]))
        for h in range(H):
            oh, lh = head_forward(q[b, :, h], kb[:, h], vb[:, h], scale, False)
            o[b, 0, h] = oh[0] if len(oh) else 0.0
            lse[b, h] = lh[0]
    return o, lse


# ---------------------------------------------------------------- grouped-query attention

def gqa_forward(q, k, v, scale: float, causal: bool):
    """Grouped-query attention ("Using it, the real way": fewer key-value heads,
    shared in groups): query head h uses K/V head h // (Hq / Hkv).
    q [B, N, Hq, d], k/v [B, N, Hkv, d] -> (o [B, N, Hq, d], lse [B, Hq, N])."""
    B, N, Hq, d = q.shape
    group = Hq // k.shape[2]
    o = np.zeros((B, N, Hq, v.shape[-1]))
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            oh, lh = head_forward(q[b, :, h], k[b, :, h // group], v[b, :, h // group], scale, causal)
            o[b, :, h] = oh
            lse[b, h] = lh
    return o, lse


def gqa_backward(q, k, v, do, scale: float, causal: bool):
    """Gradients of gqa_forward: dK and dV of a K/V head sum over its query heads."""
    B, N, Hq, d = q.shape
    group = Hq // k.shape[2]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            gq, gk, gv = head_backward(q[b, :, h], k[b, :, h // group], v[b, :, h // group], do[b, :, h], scale, causal)
            dq[b, :, h] = gq
            dk[b, :, h // group] += gk
            dv[b, :, h // group] += gv
    return dq, dk, dv


def gqa_decode_forward(q, k_cache, v_cache, scale: float):
    """Single-query decode with grouped K/V heads: q [B, 1, Hq, d], caches [B, L, Hkv, d]."""
    B, _, Hq, d = q.shape
    group = Hq // k_cache.shape[2]
    o = np.zeros((B, 1, Hq, v_cache.shape[-1]))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hq):
            oh, lh = head_forward(q[b, :, h], k_cache[b, :, h // group], v_cache[b, :, h // group], scale, False)
            o[b, 0, h] = oh[0]
            lse[b, h] = lh[0]
    return o, lse
