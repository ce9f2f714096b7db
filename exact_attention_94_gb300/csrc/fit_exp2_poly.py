"""Fit the cubic used by the software exp2 of the attention kernels.

2^x = 2^floor(x) * 2^f with f = x - floor(x) in [0, 1).  The factor 2^f is
approximated by p(f) = 1 + c1 f + c2 f^2 + c3 f^3 (c0 = 1 keeps integer x
exact).  The coefficients minimise the largest relative error over a dense
grid of [0, 1]: a discrete Chebyshev (minimax) fit solved as a linear program
(minimise t subject to |p(f_i) - 2^f_i| <= t 2^f_i), the classical LP
formulation of best uniform approximation.  Run it to regenerate the constants
printed into fa_fwd.cu:

    python fit_exp2_poly.py
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree=3, n_grid=4001):
    f = np.linspace(0.0, 1.0, n_grid)
    y = np.exp2(f)
    # unknowns: c1..c_deg, t
    powers = np.stack([f ** k for k in range(1, degree + 1)], 1)
    # p(f) - y <= t*y  ->  powers.c - t*y <= y - 1
    # y - p(f) <= t*y  -> -powers.c - t*y <= 1 - y
    a_ub = np.vstack([np.hstack([powers, -y[:, None]]), np.hstack([-powers, -y[:, None]])])
    b_ub = np.concatenate([y - 1.0, 1.0 - y])
    cost = np.zeros(degree + 1)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * (degree + 1), method="highs")
    assert res.success, res.message
    return res.x[:degree], res.x[-1]


if __name__ == "__main__":
    c, err = fit()
    print("c1..c3 =", ", ".join(f"{x:.9e}" for x in c), " max rel err =", f"{err:.3e}")
