"""Pins of the oracle's Hessian factors ("BaKron: Efficient Quantization
with Kronecker-Factored Hessians", Sec. 4.2, App. A.2 and App. D): hand-worked
values, closed forms, the Van Loan-Pitsianis rearrangement computed
explicitly from the Kronecker sum, and planted mistakes."""

import json
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hessian.json")))


def test_gram_golden():
    for c in GOLDEN["gram"]:
        G = O.weighted_gram(np.array(c["X"], float), None if c["w"] is None else np.array(c["w"], float))
        assert np.allclose(G, np.array(c["gram"]), rtol=0, atol=1e-15), c["derivation"]


def test_shampoo_one_step_golden():
    c = GOLDEN["shampoo_one_step"]
    A, B = O.shampoo_factors(np.array(c["a"], float), np.array(c["b"], float), 1)
    assert np.allclose(A, np.array(c["A"]), atol=1e-15) and np.allclose(B, np.array(c["B"]), atol=1e-15), c["derivation"]
    # the one-step weights are the squared norms
    assert np.array_equal(O.squared_norms(np.array(c["b"], float)), np.array([9.0, 1.0]))


def test_damp_golden():
    c = GOLDEN["damp"]
    assert np.array_equal(O.damp(np.array(c["G"], float), c["rel"]), np.array(c["damped"], float)), c["derivation"]


def test_orthogonal_rows_give_a_diagonal_gram():
    # rows of a 4 x 8 Hadamard block: orthogonal, squared norm 8 each
    H2 = np.array([[1, 1], [1, -1]])
    H8 = np.kron(np.kron(H2, H2), H2)
    X = 3.0 * H8[:4]
    G = O.weighted_gram(X)
    assert np.allclose(G, np.diag(np.full(4, 9.0)), atol=1e-14)


def test_single_sample_is_its_outer_product():
    x = np.array([[1.5], [-2.0], [0.25]])
    assert np.allclose(O.weighted_gram(x, [4.0]), 4.0 * np.outer(x[:, 0], x[:, 0]), atol=0)


def _rearranged(a, b):
    """R(H) of H = E[a a^T (x) b b^T] (n m x n m), rearranged explicitly:
    R(H)[(i, j), (k, l)] = H[i m + k, j m + l], rows vec(block index),
    columns vec(entry within the m x m block)."""
    n, N = a.shape
    m = b.shape[0]
    H = sum(np.kron(np.outer(a[:, t], a[:, t]), np.outer(b[:, t], b[:, t])) for t in range(N)) / N
    R = H.reshape(n, m, n, m).transpose(0, 2, 1, 3).reshape(n * n, m * m)
    return H, R


def test_shampoo_is_power_iteration_on_the_rearranged_hessian():
    rng = np.random.default_rng(0)
    n, m, N = 3, 4, 9
    a = rng.standard_normal((n, N))
    b = rng.standard_normal((m, N))
    H, R = _rearranged(a, b)
    # one step: vec(A1) = R vec(I_m), vec(B1) = R^T vec(I_n)
    A1, B1 = O.shampoo_factors(a, b, 1)
    assert np.allclose(A1.reshape(-1), R @ np.eye(m).reshape(-1), atol=1e-12)
    assert np.allclose(B1.reshape(-1), R.T @ np.eye(n).reshape(-1), atol=1e-12)
    # two steps continue from the previous iterate
    A2, B2 = O.shampoo_factors(a, b, 2)
    assert np.allclose(A2.reshape(-1), R @ B1.reshape(-1), atol=1e-10)
    assert np.allclose(B2.reshape(-1), R.T @ A1.reshape(-1), atol=1e-10)
    # many steps: the top singular pair of R(H), the best Kronecker approximation
    U, S, Vt = np.linalg.svd(R)
    A8, B8 = O.shampoo_factors(a, b, 8)
    cos = lambda x, y: abs(x @ y) / np.linalg.norm(x) / np.linalg.norm(y)  # noqa: E731
    assert cos(A8.reshape(-1), U[:, 0]) > 1 - 1e-6 and cos(B8.reshape(-1), Vt[0]) > 1 - 1e-6
    # and it fits H at least as well as the K-FAC product (both optimally scaled)
    def fit(A, B):
        K = np.kron(A, B)
        return np.linalg.norm(H - (np.sum(H * K) / np.sum(K * K)) * K)
    assert fit(A8, B8) <= fit(*O.kfac_factors(a, b)) + 1e-12


def test_both_factorizations_are_exact_for_a_fixed_output_side():
    """b_t = b for every sample: H = E[a a^T] (x) b b^T is itself a Kronecker
    product, which both approximations reproduce up to a scalar."""
    rng = np.random.default_rng(1)
    a = rng.standard_normal((3, 7))
    b = np.tile(rng.standard_normal((2, 1)), (1, 7))
    H, _ = _rearranged(a, b)
    for A, B in (O.kfac_factors(a, b), O.shampoo_factors(a, b, 1)):
        K = np.kron(A, B)
        c = np.sum(H * K) / np.sum(K * K)
        assert np.allclose(H, c * K, atol=1e-12)


def test_hessian_pins_catch_planted_mistakes(monkeypatch):
    import oracle.hessian as OH

    c = GOLDEN["gram"][1]
    X, w = np.array(c["X"], float), np.array(c["w"], float)
    # weights applied per feature instead of per sample: a shape error or a wrong value
    with pytest.raises(ValueError):
        (X * w[:, None]) @ X.T  # noqa: B018
    # a sum instead of a mean in the damping
    wrong = np.array(GOLDEN["damp"]["G"], float) + 0.5 * np.trace(np.array(GOLDEN["damp"]["G"], float)) * np.eye(2)
    assert not np.array_equal(wrong, np.array(GOLDEN["damp"]["damped"], float))
    # Shampoo weighting a_t a_t^T by its own norm instead of the output side's
    rng = np.random.default_rng(0)
    a, b = rng.standard_normal((3, 9)), rng.standard_normal((4, 9))
    _, R = _rearranged(a, b)
    with monkeypatch.context() as mp:
        mp.setattr(OH, "shampoo_factors",
                   lambda a_, b_, it=1: (OH.weighted_gram(a_, OH.squared_norms(a_)), OH.weighted_gram(b_, OH.squared_norms(b_))))
        A1, _ = OH.shampoo_factors(a, b)
        assert not np.allclose(A1.reshape(-1), R @ np.eye(4).reshape(-1), atol=1e-6)
