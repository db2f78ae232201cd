"""The GPU tests' tolerance formulas (tests/tolerances.py), checked on the CPU
against quantities they must bound or reproduce."""

import numpy as np

import oracle as O
from tolerances import check_factor, cond1, distortion_tolerance, factor_tolerance
from workloads import random_problem, toeplitz_ar1


def test_cond1_estimate_is_close_to_the_exact_condition_number():
    for H in (toeplitz_ar1(60, 0.9), random_problem(40, 50, seed=2).A.astype(np.float64), np.diag([1.0, 4.0, 1e3])):
        exact = np.linalg.cond(H, 1)
        est = cond1(H)
        assert exact / 3.0 <= est <= exact * 1.0000001, (est, exact)


def test_factor_check_accepts_the_fp32_rounding_and_rejects_a_planted_error():
    H = toeplitz_ar1(64, 0.9)
    R = O.normalized_inv_cholesky(H)
    check_factor(R.astype(np.float32), R, H)  # one rounding to fp32 is inside the bound
    G = R.astype(np.float32)
    tol = factor_tolerance(R, H)
    G[40, 3] += np.float32(4 * tol[40, 3] + 1e-6)
    try:
        check_factor(G, R, H)
    except AssertionError:
        return
    raise AssertionError("a planted error of four bounds was accepted")


def test_distortion_tolerance_covers_the_fp32_rounding_of_s_times_v():
    p = random_problem(30, 40, bits=4, seed=9)
    Vo, Wqo, _ = O.bakron(p.W, p.A, p.B, p.scales, p.bits)
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    Wq32 = (p.scales[:, None] * Vo.astype(np.float32)).astype(np.float32)
    d32 = O.distortion(p.W, Wq32.astype(np.float64), p.A, p.B)
    assert abs(d32 - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, p.B, 0.0)
    # a zero-distortion case: W already on the grid
    W = (p.scales[:, None] * Vo).astype(np.float32)
    assert distortion_tolerance(0.0, W, p.A, p.B, 0.0) > 0.0
