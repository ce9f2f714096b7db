"""Work accounting for the attention calls (host arithmetic only).

FLOP convention: a forward pass does two products per score, Q K^T and P V,
each 2*d FLOPs per score, i.e. 4*B*H*N^2*d for a dense batch; causal masking
halves it (exactly 1/2, the benchmark convention).  The backward pass is
counted as 2.5x the forward (five products instead of two).

The per-tile cost model of FlashAttention-2 ("Fewer non-matmul FLOPs",
zerotofrontier.app efficient-attention/flash-2-3) weights each of about five
non-matmul operations per score 16x: 16*5*Br*Bc / (4*Br*Bc*d) = 20/d, which is
31% at d=64 and 16% at d=128 (the displayed formula was lost in extraction;
these two printed values pin this reading).
"""
from __future__ import annotations

from typing import Iterable


def fwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    return 2.5 * fwd_flops(B, H, N, d, causal)


def varlen_fwd_flops(lengths: Iterable[int], H: int, d: int, causal: bool) -> float:
    return sum(fwd_flops(1, H, int(L), d, causal) for L in lengths)


def varlen_scores(lengths: Iterable[int]):
    """(padded, useful) score counts per head for a batch of lengths: padding
    to the longest costs B*max(L)^2, packing costs sum(L^2) ("Variable-length
    batches without padding")."""
    lengths = [int(x) for x in lengths]
    return len(lengths) * max(lengths) ** 2, sum(x * x for x in lengths)


def fa2_grid(B: int, H: int, N: int, block_rows: int):
    """FlashAttention-2 launch grid: (query blocks) x (batch * heads)
    ("Parallelism over the sequence")."""
    return -(-N // block_rows), B * H


def nonmatmul_share(d: int, ops_per_score: int = 5, weight: int = 16) -> float:
    return weight * ops_per_score / (4.0 * d)


def idle_fraction(n_blocks: int, n_sm: int) -> float:
    """Fraction of SMs left idle when fewer blocks than SMs are launched
    (FlashAttention-1's (sequence, head) grid, "Not enough parallel work")."""
    return max(0.0, 1.0 - n_blocks / n_sm)


def decode_bytes(B: int, H: int, L: int, d: int, elem_bytes: int = 2) -> float:
    """K and V cache bytes a decode step must stream once."""
    return 2.0 * B * H * L * d * elem_bytes


def masked_visible_scores(n_q: int, n_k: int, window_left: int, window_right: int) -> int:
    """Scores a bottom-right aligned mask leaves visible in one head: query i
    sees keys [i + n_k - n_q - window_left, i + n_k - n_q + window_right]
    clipped to the keys, a bound of -1 leaving its side open."""
    total = 0
    off = n_k - n_q
    for i in range(n_q):
        lo = 0 if window_left < 0 else max(0, i + off - window_left)
        hi = n_k if window_right < 0 else min(n_k, i + off + window_right + 1)
        total += max(0, hi - lo)
    return total


def masked_fwd_flops(B: int, H: int, n_q: int, n_k: int, d: int, window_left: int, window_right: int) -> float:
    """Forward FLOPs over the visible scores only (two products of 2d each);
    unlike fwd_flops' causal convention this counts the diagonal exactly."""
    return 4.0 * d * B * H * masked_visible_scores(n_q, n_k, window_left, window_right)
