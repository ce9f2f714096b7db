"""Runs one named workload a few times on cuda:0 (for profilers).

    python -m exact_attention_94_gb300.cases decode --batch 4 --iters 4
    python -m exact_attention_94_gb300.cases long --iters 3
    python -m exact_attention_94_gb300.cases varlen --iters 3
    python -m exact_attention_94_gb300.cases fp8 --iters 3      (quantise + e4m3 forward, long shape)
    python -m exact_attention_94_gb300.cases window --iters 3   (4096-key causal window, fwd + bwd)
    python -m exact_attention_94_gb300.cases prefill --iters 3  (chunked prefill forward)

Inputs are the seeded synthetic tensors of the benchmark workloads; the batch
of the decode case can be reduced so that a profiler's save and restore of
device memory stays small.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402
from exact_attention_94_gb300 import ops  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["long", "mid", "varlen", "decode", "fp8", "window", "prefill"])
    ap.add_argument("--batch", type=int, default=0, help="override the batch (dense, decode)")
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args(argv)
    w = synth.WORKLOADS["long" if a.case == "fp8" else a.case]
    B = a.batch or w.B
    if a.case == "fp8":
        x = synth.make_dense(B, w.H, w.N, w.d, seed=w.seed, k_boost=w.k_boost, device="cuda", with_do=False)
        signs = synth.hadamard_signs(w.d, 0).cuda()
        for _ in range(a.iters):
            ops.fwd_fp8(x["q"], x["k"], x["v"], signs, causal=True)
    elif a.case == "window":
        x = synth.make_dense(B, w.H, w.N, w.d, seed=0, device="cuda")
        for _ in range(a.iters):
            o, lse = ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window)
            ops.bwd_masked(x["q"], x["k"], x["v"], o, lse, x["do"], window=w.window)
    elif a.case == "prefill":
        x = synth.make_masked(B, w.N, w.n_k, w.H, w.h_kv, w.d, seed=0, device="cuda", with_do=False)
        for _ in range(a.iters):
            ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window)
    elif a.case == "decode":
        x = synth.make_decode(B, w.H, w.N, w.d, seed=0, device="cuda")
        for _ in range(a.iters):
            ops.decode(x["q"], x["k"], x["v"])
    elif a.case == "varlen":
        lengths = synth.varlen_lengths(w.B, w.len_lo, w.len_hi, w.seed)
        x = synth.make_varlen(lengths, w.H, w.d, seed=0, device="cuda")
        cu = x["cu_seqlens"].cuda()
        for _ in range(a.iters):
            o, lse = ops.fwd_varlen(x["q"], x["k"], x["v"], cu, int(lengths.max()), causal=True)
            ops.bwd_varlen(x["q"], x["k"], x["v"], o, lse, x["do"], cu, int(lengths.max()), causal=True)
    else:
        x = synth.make_dense(B, w.H, w.N, w.d, seed=0, k_boost=w.k_boost, device="cuda")
        for _ in range(a.iters):
            o, lse = ops.fwd(x["q"], x["k"], x["v"], causal=w.causal)
            ops.bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=w.causal)
    torch.cuda.synchronize()
    err = ops.device_error()
    print(f"{a.case}: {a.iters} iterations, device error {err}")
    return 0 if err == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
