"""fa_bwd_noalloc: the backward pass for callers that may not allocate device
memory (no cudaMalloc, no allocating library routine) while they issue work.

It must give the same gradients as fa_bwd with a caller-allocated workspace,
call after call.  The built-in scratch keeps the previous call's contents, so
consecutive calls here solve different problems (another seed, head count,
length and head dim, a larger problem after a smaller one and the reverse):
stale accumulator rows or per-row sums of the previous call would show up as
wrong gradients.  A problem larger than the fixed scratch is refused without
launching anything.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from exact_attention_94_gb300 import _lib, ops
from tests.parity import assert_grad

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(q, k, v, o, lse, do, causal, scale, dq, dk, dv):
    B, N, H, d = q.shape
    return _lib.load().fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(dq), _p(dk), _p(dv),
                                      B, H, N, d, int(causal), scale, _stream())


def _problem(B, H, N, d, causal, seed):
    """Inputs, the forward's o and lse, and fa_bwd's gradients (own workspace)."""
    x = synth.make_dense(B, H, N, d, seed=seed, k_boost=3.0, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse = ops.fwd(q, k, v, causal=causal)
    ref = ops.bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    return (q, k, v, o, lse, do), ref


# Two orders of three different problems: growing, and shrinking.
SEQUENCES = {
    "small_then_large": [(1, 2, 300, 64, True, 41), (2, 3, 777, 64, False, 42), (1, 4, 1000, 128, True, 43)],
    "large_then_small": [(1, 4, 1000, 128, True, 44), (2, 3, 777, 64, False, 45), (1, 2, 129, 128, False, 46)],
}


@pytest.mark.parametrize("order", sorted(SEQUENCES))
def test_noalloc_matches_workspace_backward_on_consecutive_problems(order):
    probs = [(shape, *_problem(*shape)) for shape in SEQUENCES[order]]
    # warm-up call: the first call on a device may load the library's kernels
    (B, H, N, d, causal, _), (q, k, v, o, lse, do), _ = probs[0]
    g = tuple(torch.empty_like(q) for _ in range(3))
    assert _noalloc(q, k, v, o, lse, do, causal, 1.0 / np.sqrt(d), *g) == _lib.FA_OK
    torch.cuda.synchronize()
    for call, ((B, H, N, d, causal, _), (q, k, v, o, lse, do), ref) in enumerate(probs):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        torch.cuda.synchronize()
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        free_before = torch.cuda.mem_get_info()[0]
        st = _noalloc(q, k, v, o, lse, do, causal, 1.0 / np.sqrt(d), dq, dk, dv)
        torch.cuda.synchronize()
        after = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        free_after = torch.cuda.mem_get_info()[0]
        assert st == _lib.FA_OK, _lib.status_string(st)
        assert after == before          # nothing allocated through torch
        assert free_after >= free_before  # nor anywhere else on the device (cudaMalloc, async pools)
        assert ops.device_error() == 0
        for name, gg, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert_grad(synth.to_f64(gg), synth.to_f64(r), f"{order} call {call} {name}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, H, d = 1, 32, 128
    N = 4096  # 32 x 4096 rows x (128 * 4 + 8) bytes > 32 MiB
    assert lib.fa_bwd_workspace_bytes(B, H, N, d) > _lib.FA_BWD_NOALLOC_SCRATCH_BYTES
    q = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = _noalloc(q, q, q, q, lse, q, True, 0.088, q, q, q)
    assert st == _lib.FA_ERR_SCRATCH_LIMIT
    assert _lib.status_string(st) == "FA_ERR_SCRATCH_LIMIT"
