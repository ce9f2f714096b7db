"""Work accounting pinned to the worked numbers the pages print."""
import json
import os
import pytest

from exact_attention_94_gb300 import accounting as acc

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_numbers.json")))


def test_fa2_grid():
    g = G["fa2_grid"]
    qb, bh = acc.fa2_grid(g["B"], g["H"], g["N"], g["Br"])
    assert (qb, bh, qb * bh) == (g["q_blocks"], g["bh"], g["total"])


def test_fa1_idle_fraction():
    g = G["fa1_idle"]
    assert round(100 * acc.idle_fraction(g["blocks"], g["n_sm"])) == g["idle_percent_rounded"]


def test_nonmatmul_share():
    g = G["nonmatmul_share"]
    assert round(100 * acc.nonmatmul_share(64)) == g["d64_percent_rounded"]
    assert round(100 * acc.nonmatmul_share(128)) == g["d128_percent_rounded"]


def test_varlen_scores():
    g = G["varlen_scores"]
    padded, useful = acc.varlen_scores(g["lengths"])
    assert round(padded / 1e6) == g["padded_millions_rounded"]
    assert round(useful / 1e6) == g["useful_millions_rounded"]


def test_matmul_flops_per_score():
    g = G["exp_vs_matmul_h100"]
    # a 1 x 1 "tile" at d: 4*d FLOPs per score
    assert acc.fwd_flops(1, 1, 1, g["d"], False) == g["matmul_flops_per_score"]


def test_flop_conventions():
    # long workload: B2 H16 N8192 d128 causal -> 549.8 GFLOP forward, 2.5x backward
    f = acc.fwd_flops(2, 16, 8192, 128, True)
    assert abs(f - 549.755813888e9) < 1
    assert acc.bwd_flops(2, 16, 8192, 128, True) == 2.5 * f
    assert acc.decode_bytes(64, 32, 32768, 128) == 2 * 64 * 32 * 32768 * 128 * 2


@pytest.mark.parametrize("nq,nk,wl,wr", [(10, 10, -1, 0), (7, 30, 4, 1), (30, 7, -1, 0), (16, 16, -1, -1),
                                         (50, 50, 9, 0), (12, 40, 3, -1), (5, 5, 0, 0)])
def test_masked_visible_scores_count_the_oracle_mask(nq, nk, wl, wr):
    import oracle
    assert acc.masked_visible_scores(nq, nk, wl, wr) == int(oracle.window_visible(nq, nk, wl, wr).sum())


def test_masked_flops_square_causal():
    # the exact count includes the diagonal: N (N + 1) / 2 scores
    assert acc.masked_fwd_flops(1, 1, 8, 8, 4, -1, 0) == 4 * 4 * 36
