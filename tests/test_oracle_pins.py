"""Pins of the fp64 oracle to facts fixed by the paper and by mathematics.

Source: "BaKron: Efficient Quantization with Kronecker-Factored Hessians".
Each test names what pins what.  No value here comes from the CUDA library.
"""

import itertools
import json
import os

import numpy as np
import pytest

import oracle as O
from oracle.antidiag import antidiagonal_indices
from workloads import make_config, random_problem, toeplitz_ar1

from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


SOLVERS = ["definition", "antidiagonal", "alg6", "recursive1", "recursive2", "recursive64"]


def _solve(p, method, LA=None, LB=None):
    if LA is None:
        LA, LB = O.factors_of(p.A, p.B)
    if method.startswith("recursive"):
        leaf = int(method[len("recursive"):])
        return O.bakron(p.W, LA=LA, LB=LB, scales=p.scales, bits=p.bits, method="recursive", leaf=leaf)
    return O.bakron(p.W, LA=LA, LB=LB, scales=p.scales, bits=p.bits, method=method)


# ---------------------------------------------------------------- quantizer


def test_quantizer_golden_ties_and_clamps():
    """Sec. 3.1 alphabet + round-half-even ties: hand-chosen float32-exact values."""
    for case in _golden("quantizer_ties.json")["cases"]:
        x = np.array(case["x"], dtype=np.float64)
        s = np.float32(case["s"]) if case["bits"] else None
        v, e = O.quantize(x, s, case["bits"])
        assert v.tolist() == case["v"], case
        sv = (1.0 if s is None else float(s)) * v
        assert np.allclose(e, sv - x, rtol=0, atol=0)


def test_alphabet_bounds():
    assert O.alphabet_bounds(0) is None
    assert O.alphabet_bounds(2) == (-2, 1)
    assert O.alphabet_bounds(3) == (-4, 3)
    assert O.alphabet_bounds(4) == (-8, 7)
    assert O.alphabet_bounds(8) == (-128, 127)
    with pytest.raises(ValueError):
        O.alphabet_bounds(1)


# ---------------------------------------------------------------- factors


def test_factor_2x2_golden():
    g = _golden("factor_2x2.json")
    H = np.array(g["H"])
    assert np.allclose(O.normalized_inv_cholesky(H), g["Lhat"], atol=1e-15)
    assert np.allclose(O.rev_cholesky(H), g["RevCholesky"], atol=1e-15)


def test_factor_ar1_closed_form():
    """rho^|i-j| has a tridiagonal inverse whose Cholesky factor is lower
    bidiagonal with constant ratio: L-hat = I - rho * (subdiagonal shift).
    A transposed, reversed or non-inverted factor fails this."""
    for d, rho in [(2, 0.5), (7, 0.9), (33, -0.3)]:
        L = O.normalized_inv_cholesky(toeplitz_ar1(d, rho))
        expect = np.eye(d) - rho * np.eye(d, k=-1)
        assert np.allclose(L, expect, atol=1e-12)


def test_factor_properties_random_spd():
    """Cholesky(H^-1) = RevCholesky(H)^-1: L-hat diag(1/R_jj^2) L-hat^T = H^-1, R^T R = H."""
    rng = np.random.default_rng(5)
    for d in (1, 2, 5, 16, 40):
        X = rng.standard_normal((d, 3 * d + 2))
        H = X @ X.T / X.shape[1] + 0.1 * np.eye(d)
        Lh = O.normalized_inv_cholesky(H)
        R = O.rev_cholesky(H)
        assert np.allclose(np.triu(Lh, 1), 0) and np.allclose(np.diag(Lh), 1)
        assert np.allclose(np.triu(R, 1), 0) and np.all(np.diag(R) > 0)
        assert np.allclose(R.T @ R, H, atol=1e-12)
        Hinv = np.linalg.inv(H)
        assert np.allclose(Lh @ np.diag(1.0 / np.diag(R) ** 2) @ Lh.T, Hinv, atol=1e-10)
        assert np.allclose(Lh, np.linalg.inv(R) @ np.diag(np.diag(R)), atol=1e-10)


# ---------------------------------------------------------------- worked examples


@pytest.mark.parametrize("method", ["naive"] + SOLVERS)
def test_gptq_1x2_golden(method):
    g = _golden("gptq_1x2.json")
    p = random_problem(1, 2, bits=0, seed=0)
    p.W, p.A, p.B = np.array(g["W"]), np.array(g["A"]), np.array(g["B"])
    V, Wq, E = O.bakron(p.W, p.A, p.B, None, 0, method="naive") if method == "naive" else _solve(p, method)
    assert V.tolist() == g["V"]
    assert np.allclose(E, g["E"], atol=1e-12)
    assert abs(O.distortion(p.W, Wq, p.A, p.B) - g["distortion"]) < 1e-12


@pytest.mark.parametrize("method", ["naive"] + SOLVERS)
def test_bakron_2x2_golden(method):
    g = _golden("bakron_2x2.json")
    p = random_problem(2, 2, bits=0, seed=0)
    p.W, p.A, p.B = np.array(g["W"]), np.array(g["A"]), np.array(g["B"])
    V, Wq, E = O.bakron(p.W, p.A, p.B, None, 0, method="naive") if method == "naive" else _solve(p, method)
    assert V.tolist() == g["V"]
    assert np.allclose(E, g["E"], atol=1e-12)


# ---------------------------------------------------------------- brute force


@pytest.mark.parametrize("m,n", [(1, 1), (1, 6), (6, 1), (2, 3), (3, 5), (5, 4), (7, 7)])
@pytest.mark.parametrize("bits", [0, 2, 3])
def test_naive_equals_babai_nearest_plane(m, n, bits):
    """Sec. 3.2: GPTQ on vec(W) is Babai's nearest plane in the basis
    RevCholesky(A (x) B) -- an independent formulation (no error feedback)."""
    p = random_problem(m, n, bits=bits, seed=10 * m + n + bits)
    Vn, _, En = O.bakron_naive(p.W, p.A, p.B, p.scales, p.bits)
    Vb, Eb = O.babai_nearest_plane(p.W, p.A, p.B, p.scales, p.bits)
    assert np.array_equal(Vn, Vb)
    assert np.allclose(En, Eb, atol=1e-12)


@pytest.mark.parametrize("m,n", list(itertools.product([1, 2, 3, 5, 8], [1, 2, 4, 7])))
@pytest.mark.parametrize("bits,kind", [(0, "gram"), (2, "gram"), (4, "gram"), (3, "ar1")])
def test_theorem_3_2_all_solvers_agree_with_naive(m, n, bits, kind):
    """Theorem 3.2: naive, antidiagonal, recursive and BaKron give one output."""
    p = random_problem(m, n, bits=bits, seed=100 * m + n, kind=kind)
    Vn, _, En = O.bakron_naive(p.W, p.A, p.B, p.scales, p.bits)
    for method in SOLVERS:
        V, Wq, E = _solve(p, method)
        assert np.array_equal(V, Vn), method
        assert np.allclose(E, En, atol=1e-11), method


def test_c1_naive_equals_recursive():
    """Workload c1 (64 x 64, alphabet Z): the 4096 x 4096 Kronecker system."""
    p = make_config("c1")
    Vn, _, En = O.bakron_naive(p.W, p.A, p.B, p.scales, p.bits)
    V, _, E = O.bakron(p.W, p.A, p.B, p.scales, p.bits)
    assert np.array_equal(V, Vn)
    assert np.abs(E - En).max() < 1e-10


def test_c2_leaf_and_split_independence():
    """Workload c2: recursion with 64- and 16-entry leaves (different blocking
    and rounding order of the products) gives the same codes."""
    p = make_config("c2")
    LA, LB = O.factors_of(p.A, p.B)
    V1, _, E1 = O.bakron(p.W, LA=LA, LB=LB, scales=p.scales, bits=p.bits, leaf=64)
    V2, _, E2 = O.bakron(p.W, LA=LA, LB=LB, scales=p.scales, bits=p.bits, leaf=16)
    assert np.array_equal(V1, V2)
    assert np.abs(E1 - E2).max() < 1e-12


# ---------------------------------------------------------------- special cases


@pytest.mark.parametrize("m,n,bits", [(4, 9, 3), (9, 4, 0), (16, 16, 4)])
def test_identity_b_is_rowwise_gptq(m, n, bits):
    """B = I: the Hessian X X^T (x) I of GPTQ (Sec. 1); every row is Algorithm 1 with H = A."""
    p = random_problem(m, n, bits=bits, seed=7, kind="identity_b")
    Vg, _, Eg = O.gptq_rows(p.W, p.A, p.scales, p.bits)
    for method in ["antidiagonal", "recursive1", "recursive64", "alg6"]:
        V, _, E = _solve(p, method)
        assert np.array_equal(V, Vg), method
        assert np.allclose(E, Eg, atol=1e-12)


@pytest.mark.parametrize("m,n,bits", [(5, 3, 2), (8, 8, 4), (3, 11, 0)])
def test_diagonal_factors_are_round_to_nearest(m, n, bits):
    """A, B diagonal: L-hat = I, so every entry is rounded on its own."""
    p = random_problem(m, n, bits=bits, seed=3, kind="diagonal")
    W32 = p.W.astype(np.float32)
    y = W32 if p.scales is None else (W32 / p.scales[:, None]).astype(np.float32)
    rtn = np.rint(y)
    if bits:
        rtn = np.clip(rtn, -(1 << (bits - 1)), (1 << (bits - 1)) - 1)
    for method in ["naive"] + SOLVERS:
        V = O.bakron(p.W, p.A, p.B, p.scales, p.bits, method="naive")[0] if method == "naive" else _solve(p, method)[0]
        assert np.array_equal(V, rtn.astype(np.int64)), method


@pytest.mark.parametrize("bits", [0, 3])
def test_ar1_output_factor_is_first_order_error_feedback(bits):
    """A = I, B = rho^|i-j|: L-hat_B = I - rho S, so each column is the
    first-order error-feedback (noise-shaping) quantizer
    x_p = W_pq - rho e_(p-1), v_p = q(x_p), e_p = s_p v_p - x_p."""
    rho = 0.9
    p = random_problem(12, 5, bits=bits, seed=11, kind="ar1")
    V, _, E = _solve(p, "recursive64")
    W = p.W.astype(np.float64)
    for q in range(p.n):
        prev = 0.0
        for r in range(p.m):
            x = W[r, q] - rho * prev
            v, e = O.quantize(x, None if p.scales is None else p.scales[r], bits)
            assert V[r, q] == v
            prev = float(e)


def test_on_alphabet_input_is_fixed_point():
    """W already on the alphabet: every error is zero and V = W."""
    p = random_problem(6, 9, bits=3, seed=2)
    p.scales = np.ones(6, dtype=np.float32)
    p.W = np.random.default_rng(0).integers(-4, 4, size=(6, 9)).astype(np.float32)
    V, Wq, E = _solve(p, "recursive64")
    assert np.array_equal(V, p.W.astype(np.int64)) and np.all(E == 0)


# ---------------------------------------------------------------- identities and bounds


@pytest.mark.parametrize("key_or_shape", ["c1", (13, 21, 3), (21, 13, 2)])
def test_exact_identities(key_or_shape):
    """App. B eq. (1): Wq - W0 = L_B E L_A^T with E the errors at rounding;
    and the distortion equals sum_ij E_ij^2 R_B,ii^2 R_A,jj^2."""
    if isinstance(key_or_shape, str):
        p = make_config(key_or_shape)
    else:
        m, n, b = key_or_shape
        p = random_problem(m, n, bits=b, seed=9)
    LA, LB = O.factors_of(p.A, p.B)
    V, Wq, E = O.bakron(p.W, LA=LA, LB=LB, scales=p.scales, bits=p.bits)
    W0 = p.W.astype(np.float64)
    assert np.abs(W0 + LB @ E @ LA.T - Wq).max() < 1e-11
    assert np.abs(O.errors_from_output(p.W, Wq, LA, LB) - E).max() < 1e-10
    d1 = O.distortion(p.W, Wq, p.A, p.B)
    d2 = O.distortion_from_errors(E, p.A, p.B)
    assert abs(d1 - d2) <= 1e-10 * abs(d1)


def test_corollary_3_4_bound_c1():
    """Corollary 3.4 for the alphabet Z (workload c1): every |E_ij| <= 1/2 and
    the distortion stays below 1/4 sum R_B,ii^2 R_A,jj^2 <= 1/4 tr A tr B."""
    p = make_config("c1")
    V, Wq, E = O.bakron(p.W, p.A, p.B, None, 0)
    assert np.abs(E).max() <= 0.5
    inner, outer = O.corollary34_bound(p.A, p.B)
    d = O.distortion(p.W, Wq, p.A, p.B)
    assert d <= inner <= outer


def test_errors_bounded_by_half_step_unclamped():
    """Every unclamped code is a nearest rounding: |E_ij| <= s_i / 2."""
    p = random_problem(24, 31, bits=4, seed=4)
    V, _, E = O.bakron(p.W, p.A, p.B, p.scales, p.bits)
    inner = (V > -8) & (V < 7)
    lim = 0.5 * p.scales.astype(np.float64)[:, None] * (1 + 1e-6)
    assert np.all(np.abs(E)[inner] <= np.broadcast_to(lim, E.shape)[inner])


def test_antidiagonal_indices_cover_matrix_once():
    for m, n in [(1, 1), (3, 7), (7, 3), (5, 5)]:
        seen = np.zeros((m, n), dtype=int)
        for k in range(m + n - 1):
            r, c = antidiagonal_indices(m, n, k)
            assert np.all(r + c == k)
            seen[r, c] += 1
        assert np.all(seen == 1)


# ---------------------------------------------------------------- planted mistakes


def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle and check a pin fails for each."""
    import oracle.factors as F

    good = F.normalized_inv_cholesky

    # (1) Cholesky of H instead of H^-1: the AR(1) closed form breaks.
    def chol_not_inverted(H):
        L = np.linalg.cholesky(np.asarray(H, np.float64))
        return L / np.diag(L)[None, :]

    assert not np.allclose(chol_not_inverted(toeplitz_ar1(7, 0.9)), np.eye(7) - 0.9 * np.eye(7, k=-1), atol=1e-6)

    # (2) A dropped or transposed factor in the recursive solver: naive disagrees.
    p = random_problem(5, 6, bits=3, seed=21)
    LA, LB = O.factors_of(p.A, p.B)
    Vn, _, _ = O.bakron_naive(p.W, p.A, p.B, p.scales, p.bits)
    Vdrop, _, _ = O.bakron(p.W, LA=LA, LB=np.eye(5), scales=p.scales, bits=p.bits)  # output factor dropped
    assert not np.array_equal(Vdrop, Vn)
    Vtr, _, _ = O.bakron(p.W, LA=np.triu(LA.T), LB=LB, scales=p.scales, bits=p.bits)  # transposed L_A
    assert not np.array_equal(Vtr, Vn)

    # (3) Row-major instead of column-major vec in the naive solver: differs
    # from the factored solvers (Prop. 3.1 fixes the Kronecker order).
    W = p.W.astype(np.float64)
    H_wrong = np.kron(p.B.astype(np.float64), p.A.astype(np.float64))
    Lw = good(H_wrong)
    s = np.tile(p.scales, p.n)
    codes, _, _ = O.naive.gptq_vector(W.flatten(order="F"), Lw, s, p.bits)
    assert not np.array_equal(codes.reshape((p.m, p.n), order="F"), Vn)
