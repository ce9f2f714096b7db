"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the bench.

This module holds only random-number generation and shape bookkeeping: no
attention arithmetic lives here, so neither side of a parity check can borrow
the other's maths through it.

Recipe (the same for every tensor): draw fp32 values from N(0, 1) with a
seeded ``torch.Generator`` and round them to bf16 (round to nearest even).
Each tensor has its own seed, ``seed * 100 + idx`` with idx q=0, k=1, v=2,
dO=3, sequence lengths=4.  The oracle consumes the very bf16 values the GPU
kernels see (upcast to float64 on the host).

Workloads (one line each, sizes as the pages' worked examples and the
benchmark configurations state them):

* ``tiny``    B=1  H=2  N=256  d=64, causal and non-causal
* ``mid``     B=16 H=16 N=2048 d=64, non-causal
* ``long``    B=2  H=16 N=8192 d=128, causal, K multiplied by 3 (in fp32,
  before rounding) in heads h < H/2 so that the running maximum of the online
  softmax jumps
* ``varlen``  32 sequences, lengths uniform integers in [128, 4096], packed
  end to end, H=32 d=128, causal per sequence
* ``decode``  B=64 single queries against a 32768-token KV cache, H=32 d=128
* ``window``  B=1 H=32 N=16384 d=128, causal sliding window of 4096 keys
  (window_left 4095); the pages give no size for a windowed run, so this one
  is a long-context configuration of the usual 4096-token window
* ``prefill`` chunked prefill: B=8 chunks of 2048 new queries against
  16384-key caches, 32 query heads sharing 8 K/V heads, d=128, bottom-right
  causal; sizes chosen here, the pages' example (4 queries, 128 keys) being
  a toy
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

IDX_Q, IDX_K, IDX_V, IDX_DO, IDX_LENGTHS = 0, 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "dense" | "varlen" | "decode" | "masked"
    B: int                    # batch (dense/decode) or number of sequences (varlen)
    H: int
    N: int                    # sequence length (dense), KV cache length (decode), max length (varlen)
    d: int
    causal: bool
    k_boost: float = 1.0      # multiplier on K for heads h < H/2 (1.0 = none)
    len_lo: int = 0           # varlen: inclusive length range
    len_hi: int = 0
    seed: int = 0
    n_k: int = 0              # keys per sequence when they differ from N (0 = N)
    h_kv: int = 0             # K/V heads when fewer than H (0 = H)
    window: tuple = (-1, -1)  # (window_left, window_right); (-1, 0) with causal

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    "tiny": Workload("tiny", "dense", 1, 2, 256, 64, False),
    "tiny_causal": Workload("tiny_causal", "dense", 1, 2, 256, 64, True),
    "mid": Workload("mid", "dense", 16, 16, 2048, 64, False),
    "long": Workload("long", "dense", 2, 16, 8192, 128, True, k_boost=3.0),
    "varlen": Workload("varlen", "varlen", 32, 32, 4096, 128, True, len_lo=128, len_hi=4096),
    "decode": Workload("decode", "decode", 64, 32, 32768, 128, False),
    "window": Workload("window", "masked", 1, 32, 16384, 128, True, window=(4095, 0)),
    "prefill": Workload("prefill", "masked", 8, 32, 2048, 128, True, n_k=16384, h_kv=8, window=(-1, 0)),
}


def _gen(seed: int, idx: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100 + idx)
    return g


def randn_bf16(shape, seed: int, idx: int, device: str = "cpu",
               head_dim_axis: Optional[int] = None, boost: float = 1.0,
               boost_heads: int = 0) -> torch.Tensor:
    """N(0,1) fp32 draw rounded to bf16; optionally multiply heads [0, boost_heads)
    along ``head_dim_axis`` by ``boost`` in fp32 before the rounding."""
    x = torch.randn(shape, generator=_gen(seed, idx, device), dtype=torch.float32, device=device)
    if boost != 1.0 and boost_heads > 0:
        sl = [slice(None)] * x.dim()
        sl[head_dim_axis] = slice(0, boost_heads)
        x[tuple(sl)] *= boost
    return x.to(torch.bfloat16)


def varlen_lengths(n_seqs: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Integer lengths drawn uniformly from [lo, hi] inclusive (int64, CPU)."""
    return torch.randint(lo, hi + 1, (n_seqs,), generator=_gen(seed, IDX_LENGTHS, "cpu"))


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    """[0, L1, L1+L2, ...] as int32 (length B+1)."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def make_dense(B, H, N, d, seed=0, k_boost=1.0, device="cpu", with_do=True):
    """Q, K, V (and dO) in [B, N, H, d] bf16."""
    shape = (B, N, H, d)
    out = {
        "q": randn_bf16(shape, seed, IDX_Q, device),
        "k": randn_bf16(shape, seed, IDX_K, device, head_dim_axis=2, boost=k_boost,
                        boost_heads=H // 2 if k_boost != 1.0 else 0),
        "v": randn_bf16(shape, seed, IDX_V, device),
    }
    if with_do:
        out["do"] = randn_bf16(shape, seed, IDX_DO, device)
    return out


def make_varlen(lengths, H, d, seed=0, device="cpu", with_do=True):
    """Packed Q, K, V (and dO) in [total, H, d] bf16 plus int32 cu_seqlens."""
    cu = cu_seqlens_from_lengths(lengths)
    total = int(cu[-1])
    shape = (total, H, d)
    out = {
        "q": randn_bf16(shape, seed, IDX_Q, device),
        "k": randn_bf16(shape, seed, IDX_K, device),
        "v": randn_bf16(shape, seed, IDX_V, device),
        "cu_seqlens": cu,
    }
    if with_do:
        out["do"] = randn_bf16(shape, seed, IDX_DO, device)
    return out


def make_decode(B, H, L, d, seed=0, device="cpu"):
    """q [B, 1, H, d] and a KV cache [B, L, H, d] (bf16)."""
    return {
        "q": randn_bf16((B, 1, H, d), seed, IDX_Q, device),
        "k": randn_bf16((B, L, H, d), seed, IDX_K, device),
        "v": randn_bf16((B, L, H, d), seed, IDX_V, device),
    }


def make_workload(w: Workload, device="cpu", with_do=True):
    if w.kind == "dense":
        return make_dense(w.B, w.H, w.N, w.d, w.seed, w.k_boost, device, with_do)
    if w.kind == "varlen":
        lengths = varlen_lengths(w.B, w.len_lo, w.len_hi, w.seed)
        out = make_varlen(lengths, w.H, w.d, w.seed, device, with_do)
        out["lengths"] = lengths
        return out
    if w.kind == "decode":
        return make_decode(w.B, w.H, w.N, w.d, w.seed, device)
    raise ValueError(w.kind)


def to_f64(t: torch.Tensor):
    """Exact upcast of bf16 values to a float64 numpy array (host copy)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def make_paged_decode(lengths, H, d, page_size=16, spare_pages=3, seed=0, device="cpu"):
    """A paged cache for a decode batch: each sequence b gets ceil(L_b / page_size)
    pages drawn without replacement from a shuffled pool (plus spare pages
    nobody owns); block_table rows are padded with page 0.  Page contents,
    including unused slots, are N(0,1) bf16 like every other input.
    Returns q [B,1,H,d], k_pages/v_pages [num_pages, page_size, H, d],
    block_table int32 [B, max_blocks], seq_lens int32 [B]."""
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    blocks = [-(-L // page_size) for L in lengths]
    max_blocks = max(1, max(blocks))
    num_pages = sum(blocks) + spare_pages
    perm = torch.randperm(num_pages, generator=_gen(seed, IDX_LENGTHS, "cpu"))
    table = torch.zeros((B, max_blocks), dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for j in range(blocks[b]):
            table[b, j] = int(perm[nxt])
            nxt += 1
    return {
        "q": randn_bf16((B, 1, H, d), seed, IDX_Q, device),
        "k_pages": randn_bf16((num_pages, page_size, H, d), seed, IDX_K, device),
        "v_pages": randn_bf16((num_pages, page_size, H, d), seed, IDX_V, device),
        "block_table": table,
        "seq_lens": torch.tensor(lengths, dtype=torch.int32),
    }


def make_masked(B, Nq, Nk, Hq, Hkv, d, seed=0, device="cpu", with_do=True):
    """Queries against a key/value set of another length (chunked prefill):
    q (and dO) [B, Nq, Hq, d], k, v [B, Nk, Hkv, d], bf16."""
    out = {
        "q": randn_bf16((B, Nq, Hq, d), seed, IDX_Q, device),
        "k": randn_bf16((B, Nk, Hkv, d), seed, IDX_K, device),
        "v": randn_bf16((B, Nk, Hkv, d), seed, IDX_V, device),
    }
    if with_do:
        out["do"] = randn_bf16((B, Nq, Hq, d), seed, IDX_DO, device)
    return out


def make_masked_varlen(lengths_q, lengths_k, Hq, Hkv, d, seed=0, device="cpu", with_do=True):
    """Packed queries and keys with their own lengths per sequence:
    q (and dO) [total_q, Hq, d], k, v [total_k, Hkv, d], int32 cu_seqlens_q / _k."""
    cu_q = cu_seqlens_from_lengths(lengths_q)
    cu_k = cu_seqlens_from_lengths(lengths_k)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    out = {
        "q": randn_bf16((tq, Hq, d), seed, IDX_Q, device),
        "k": randn_bf16((tk, Hkv, d), seed, IDX_K, device),
        "v": randn_bf16((tk, Hkv, d), seed, IDX_V, device),
        "cu_seqlens_q": cu_q,
        "cu_seqlens_k": cu_k,
    }
    if with_do:
        out["do"] = randn_bf16((tq, Hq, d), seed, IDX_DO, device)
    return out


IDX_SIGNS, IDX_OUTLIER_MASK, IDX_OUTLIER_VALUE = 5, 6, 7


def hadamard_signs(d: int, seed: int = 0) -> torch.Tensor:
    """The random +-1 diagonal of incoherent processing, drawn on the host:
    int8 [d] of -1 / +1 with equal probability."""
    bits = torch.randint(0, 2, (d,), generator=_gen(seed, IDX_SIGNS, "cpu"))
    return (bits * 2 - 1).to(torch.int8)


def outlier_bf16(shape, seed: int, idx: int, device: str = "cpu", frac: float = 0.001,
                 outlier_std: float = 10.0) -> torch.Tensor:
    """Entries N(0, 1) plus, on a fraction ``frac`` of them chosen independently,
    an extra N(0, outlier_std^2) term; fp32 draws rounded to bf16.  The default
    is the outlier test of the FP8 discussion (0.1% of entries, N(0, 100))."""
    base = torch.randn(shape, generator=_gen(seed, idx, device), dtype=torch.float32, device=device)
    g = _gen(seed * 7 + idx, IDX_OUTLIER_MASK, device)
    mask = torch.rand(shape, generator=g, device=device) < frac
    extra = torch.randn(shape, generator=_gen(seed * 7 + idx, IDX_OUTLIER_VALUE, device), dtype=torch.float32,
                        device=device) * outlier_std
    return (base + mask * extra).to(torch.bfloat16)
