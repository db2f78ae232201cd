"""The chunk products' precision mode, modelled on the CPU in fp32 numpy and
checked against exact rational products (no GPU; this pins the error
analysis of the tensor-core path, not the kernel itself).

A chunk product computes Y[r, q] = sum_k F[r, k] D[k, q] for a 128-deep
chunk, F an fp32 factor block and D double-float sources (E or G values of
the solve, below 2^eD = 2 sigma).  On the tensor cores it runs as bf16
integer digits (Ozaki, Ogita, Oishi and Rump, "Error-free transformations of
matrix multiplication by using fast routines of matrix multiplication and
its applications", Numer. Algorithms 2012):
  F[r, k] ~ 2^(e_r - 7) sum_{a<5} f_a 256^-a   (one exponent per row and chunk)
  D[k, q] ~ 2^(eD - 7)  sum_{b<6} d_b 256^-b   (one global exponent)
with |f_a|, |d_b| <= 128; the pairs with a + b <= 5 are summed per level
l = a + b in fp32 (exact: every level stays below 2^24) and the six levels
are combined in double-float, then rounded onto the 64-bit fixed-point grid
of unit 2^(eD - 54).  The model below takes the same steps in the same
precision and order; the tests check the exactness precondition on the
level sums and the total error against a bound derived from the digit
counts."""

from fractions import Fraction

import numpy as np
import pytest

f32 = np.float32
K = 128  # chunk depth
N_FDIG, N_SDIG, N_LEV = 5, 6, 6


def bound_exp(mx: float) -> int:
    """e with mx < 2^e <= 2 mx (frexp), as the kernels take it."""
    if not mx > 0:
        return -100
    return max(int(np.frexp(np.float32(mx))[1]), -100)


def two_sum(a, b):
    s = (a + b).astype(f32)
    bb = (s - a).astype(f32)
    e = ((a - (s - bb)).astype(f32) + (b - bb).astype(f32)).astype(f32)
    return s, e


def factor_digits(F, e_rows):
    """Five digits per entry: u = F 2^(7 - e_r), d = rint(u), u <- 256 (u - d)."""
    u = (F * np.ldexp(f32(1), 7 - e_rows).astype(f32)[:, None]).astype(f32)
    out = []
    for _ in range(N_FDIG):
        d = np.rint(u).astype(f32)
        out.append(d.astype(np.int64))
        u = ((u - d).astype(f32) * f32(256)).astype(f32)
    return out


def source_digits(hi, lo, eD):
    """Six digits of the double-float hi + lo on the global exponent eD."""
    sc = f32(2.0 ** (7 - eD))
    ux, uy = (hi * sc).astype(f32), (lo * sc).astype(f32)
    out = []
    for _ in range(N_SDIG):
        dg = np.rint(ux).astype(f32)
        out.append(dg.astype(np.int64))
        rx, ry = two_sum((ux - dg).astype(f32), uy)
        ux, uy = (rx * f32(256)).astype(f32), (ry * f32(256)).astype(f32)
    return out


def levels(fd, sd):
    """Level l = sum over digit pairs a + b = l (a < 5, b < 6, l < 6), exact integers."""
    lev = np.zeros((N_LEV, fd[0].shape[0], sd[0].shape[1]), dtype=np.int64)
    for a in range(N_FDIG):
        for b in range(N_SDIG):
            if a + b < N_LEV:
                lev[a + b] += fd[a] @ sd[b]
    return lev


def combine(lev):
    """The epilogue's double-float sum of the six levels (fp32 steps)."""
    lv = [lev[l].astype(f32) for l in range(N_LEV)]
    y, ye = two_sum(lv[0], (lv[1] * f32(2.0 ** -8)).astype(f32))
    y2, y2e = two_sum(ye, (lv[2] * f32(2.0 ** -16)).astype(f32))
    tail = ((lv[3] * f32(2.0 ** -24)).astype(f32) + (lv[4] * f32(2.0 ** -32)).astype(f32)).astype(f32)
    tail = (tail + (lv[5] * f32(2.0 ** -40)).astype(f32)).astype(f32)
    y, ye = two_sum(y, y2)
    return two_sum(y, (ye + (y2e + tail).astype(f32)).astype(f32))


def model_product(F, hi, lo, sigma):
    """Y = F (hi + lo) on the fixed-point grid, as exact Fractions, with the
    largest level magnitude seen and the grid unit."""
    e_rows = np.array([bound_exp(float(np.max(np.abs(F[r])))) for r in range(F.shape[0])])
    eD = bound_exp(sigma)
    unit_exp = max(eD, -60) - 54
    lev = levels(factor_digits(F, e_rows), source_digits(hi, lo, eD))
    ys, ye = combine(lev)
    Y = [[0] * hi.shape[1] for _ in range(F.shape[0])]
    for r in range(F.shape[0]):
        scale = Fraction(2) ** (int(e_rows[r]) + eD - 14 - unit_exp)  # levels -> fixed-point units
        for q in range(hi.shape[1]):
            fixed = round(Fraction(float(ys[r, q])) * scale) + round(Fraction(float(ye[r, q])) * scale)
            Y[r][q] = Fraction(fixed) * Fraction(2) ** unit_exp
    return Y, int(np.max(np.abs(lev))), e_rows, eD, unit_exp


def exact_product(F, hi, lo):
    Fr = [[Fraction(float(x)) for x in row] for row in F]
    Dr = [[Fraction(float(h)) + Fraction(float(l)) for h, l in zip(hr, lr)] for hr, lr in zip(hi, lo)]
    return [[sum(Fr[r][k] * Dr[k][q] for k in range(F.shape[1])) for q in range(hi.shape[1])]
            for r in range(F.shape[0])]


def error_bound(F, hi, lo, e_rows, eD, unit_exp, r, q):
    """Factor digits keep u to 2^-33 (2^(e_r - 40) per entry), source digits
    the value to 2^(eD - 48); the dropped pairs (a + b >= 6) add at most
    K sum_{l>=6} (pairs of l) 2^14 256^-l 2^(e_r + eD - 14); the double-float
    sum of the levels and the two roundings to the grid one unit each, and
    the levels' fp32 combination 2^-44 of their magnitude."""
    sF = float(np.sum(np.abs(F[r].astype(np.float64))))
    sD = float(np.sum(np.abs(hi[:, q].astype(np.float64)) + np.abs(lo[:, q].astype(np.float64))))
    dropped = sum(sum(1 for a in range(N_FDIG) for b in range(N_SDIG) if a + b == l) * 256.0 ** -l
                  for l in range(N_LEV, N_FDIG + N_SDIG - 1))
    return (2.0 ** (int(e_rows[r]) - 40) * sD + 2.0 ** (eD - 48) * sF
            + K * 2.0 ** 14 * dropped * 2.0 ** (int(e_rows[r]) + eD - 14)
            + 2.0 ** (int(e_rows[r]) + eD - 44) * K + 3 * 2.0 ** unit_exp)


def _inputs(seed, rows=6, cols=3, spread=12):
    rng = np.random.default_rng(seed)
    # factor rows spanning a few binades inside each row, as in the
    # normalized inverse Cholesky factors (|entries| <= 1)
    F = (rng.standard_normal((rows, K)) * np.exp2(-rng.integers(0, spread, (rows, K)))).astype(f32)
    F = np.clip(F, -1, 1).astype(f32)
    sigma = float(np.float32(2.0 ** rng.integers(-6, 3)))
    hi = (rng.uniform(-1, 1, (K, cols)) * sigma * 0.9).astype(f32)
    # low words below half an ulp of the high words
    lo = (rng.uniform(-0.5, 0.5, (K, cols)) * np.spacing(np.abs(hi).astype(f32))).astype(f32)
    return F, hi, lo, sigma


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_model_matches_the_exact_product_within_the_derived_bound(seed):
    F, hi, lo, sigma = _inputs(seed)
    Y, lmax, e_rows, eD, unit_exp = model_product(F, hi, lo, sigma)
    X = exact_product(F, hi, lo)
    assert lmax < 2 ** 24  # every level sum is an exact fp32 value, in any summation order
    worst = 0.0
    for r in range(F.shape[0]):
        for q in range(hi.shape[1]):
            err = abs(float(Y[r][q] - X[r][q]))
            bound = error_bound(F, hi, lo, e_rows, eD, unit_exp, r, q)
            assert err <= bound, (r, q, err, bound)
            scale = float(np.sum(np.abs(F[r].astype(np.float64)) * np.abs(hi[:, q].astype(np.float64))))
            worst = max(worst, err / scale)
    # on factor rows spanning a dozen binades the error stays near 2^-40 of
    # sum |F| |D| (the truncation of the fifth factor digit; 1.4e-13 to
    # 6.1e-13 over these seeds)
    assert worst < 2e-12, worst


def test_level_sums_stay_exact_for_extreme_digits():
    """Entries just below the block bound round their top digit to 128 and
    every digit pair to its largest magnitude with one sign: the level sums
    still stay below 2^24."""
    F = np.full((2, K), np.float32(0.99999994), dtype=f32)  # u = 127.99999 -> d_0 = 128, then -0.0...
    F[1] = -F[1]
    sigma = 1.0
    hi = np.full((K, 2), np.float32(1.9999999), dtype=f32)  # just below 2^eD = 2
    lo = np.zeros((K, 2), dtype=f32)
    _, lmax, _, _, _ = model_product(F, hi, lo, sigma)
    assert lmax < 2 ** 24, lmax
    # all-digit extremes: the largest level holds 5 pairs of 128 x 128 over K = 128
    assert 5 * 128 * 128 * K < 2 ** 24


def test_a_dropped_factor_digit_breaks_the_bound():
    """Planted mistake: four factor digits instead of five leave an error
    near 2^-32 of the row scale, above the bound the tests use."""
    global N_FDIG
    F, hi, lo, sigma = _inputs(7, rows=3, cols=2, spread=20)
    X = exact_product(F, hi, lo)
    saved = N_FDIG
    try:
        N_FDIG = 4
        Y, _, e_rows, eD, unit_exp = model_product(F, hi, lo, sigma)
    finally:
        N_FDIG = saved
    excess = [abs(float(Y[r][q] - X[r][q])) / error_bound(F, hi, lo, e_rows, eD, unit_exp, r, q)
              for r in range(F.shape[0]) for q in range(hi.shape[1])]
    assert max(excess) > 1.0, excess
