"""The lazy rescale on the device, counted ("efficient-attention/flash-2-3",
section "And on Blackwell": rescale only when the maximum has grown by enough
to threaten overflow, about 10x fewer rescales).

A test-only build of the forward kernel (FA_COUNT_RESCALES; the product
library has no counter) counts, per (batch, head), the (row, key tile) pairs
whose reference maximum moves while an earlier one existed.  The oracle's
tiled model (oracle.attention.online_head_forward, 128-key blocks, the same
rule in float64) counts the same events on the same bf16 inputs.  The kernel
decides in float32 on scores accumulated in float32, so a decision can flip
where the growth lands within rounding of the threshold: the counts must agree
to within 0.2% + 2.  Workload: the long one (B2 H16 N8192 d128, causal, K x 3
in heads 0-7); heads 0 (boosted) and 8 (plain), thresholds 8 and 0.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import _lib, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def counting_lib():
    lib = ctypes.CDLL(build.build_counting())
    for name, (res, args) in _lib.SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    lib.fa_test_rescale_counts.restype = ctypes.c_int
    lib.fa_test_rescale_counts.argtypes = [ctypes.c_void_p, ctypes.c_int]
    return lib


def test_device_rescales_match_the_oracle_model(counting_lib):
    lib = counting_lib
    w = synth.WORKLOADS["long"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=w.seed, k_boost=w.k_boost, with_do=False, device="cuda")
    q, k, v = x["q"], x["k"], x["v"]
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    counts = np.zeros(w.B * w.H, dtype=np.uint64)
    heads = [(0, 0), (0, 8)]
    ref_inputs = {bh: tuple(synth.to_f64(x[n][bh[0], :, bh[1]]) for n in ("q", "k", "v")) for bh in heads}
    seen = {}
    try:
        for tau in (8.0, 0.0):
            assert lib.fa_set_option(_lib.FA_OPT_RESCALE_TAU, tau) == _lib.FA_OK
            assert lib.fa_test_rescale_counts(counts.ctypes.data, counts.size) == 0  # clears
            st = lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), w.B, w.H, w.N, w.d, 1, w.scale, stream)
            assert st == _lib.FA_OK
            torch.cuda.synchronize()
            assert lib.fa_test_rescale_counts(counts.ctypes.data, counts.size) == 0
            for b, h in heads:
                qh, kh, vh = ref_inputs[(b, h)]
                _, _, n_ref = oracle.online_head_forward(qh, kh, vh, w.scale, True, 128, tau)
                n_gpu = int(counts[b * w.H + h])
                seen[(tau, b, h)] = (n_gpu, n_ref)
                assert abs(n_gpu - n_ref) <= 2 + 0.002 * n_ref, (tau, b, h, n_gpu, n_ref)
    finally:
        lib.fa_set_option(_lib.FA_OPT_RESCALE_TAU, 8.0)
    # the threshold's effect on the boosted head: many times fewer rescales
    assert seen[(0.0, 0, 0)][0] > 10 * seen[(8.0, 0, 0)][0]
    print("rescales (tau, b, h): (gpu, oracle model)", seen)
