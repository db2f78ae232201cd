"""Distortion and exact identities (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians":
  Sec. 4.1 / Prop. 3.1: the distortion of V is the quadratic form
  ||vec(Wq - W)||^2_{A (x) B} = tr(A (Wq - W)^T B (Wq - W)).
  App. B, eq. (1): one product L_B E L_A^T applies every elementary update of
  the entries in E's support.  Summed over all anti-diagonals, the final
  weights are Wq = W0 + L_B E L_A^T, with E the errors at rounding time.
  Sec. 3.7, Theorem 3.3 / Corollary 3.4: with R = RevCholesky,
  ||R_B (V - W) R_A^T||_F^2 <= 1/4 sum_ij R_B,ii^2 R_A,jj^2 <= 1/4 tr A tr B
  for the alphabet Z.

Derived here: L-hat = R^-1 diag(R) (Cholesky(H^-1) = RevCholesky(H)^-1),
so R_B (Wq - W) R_A^T = diag(R_B) E diag(R_A) and the distortion equals
sum_ij E_ij^2 R_B,ii^2 R_A,jj^2 exactly.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from .factors import rev_cholesky


def distortion(W, Wq, A, B) -> float:
    """tr(A (Wq - W)^T B (Wq - W)) in float64 (A, B symmetric)."""
    D = np.asarray(Wq, dtype=np.float64) - np.asarray(W, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    return float(np.sum((B @ D) * (D @ A)))


def errors_from_output(W, Wq, LA, LB) -> np.ndarray:
    """E = L_B^-1 (Wq - W) L_A^-T: the errors an output implies (two unit
    lower-triangular solves, float64)."""
    D = np.asarray(Wq, dtype=np.float64) - np.asarray(W, dtype=np.float64)
    X = solve_triangular(np.asarray(LB, dtype=np.float64), D, lower=True, unit_diagonal=True)
    Et = solve_triangular(np.asarray(LA, dtype=np.float64), X.T, lower=True, unit_diagonal=True)
    return np.ascontiguousarray(Et.T)


def distortion_from_errors(E, A, B) -> float:
    """sum_ij E_ij^2 R_B,ii^2 R_A,jj^2 with R = RevCholesky."""
    ra = np.diag(rev_cholesky(A)) ** 2
    rb = np.diag(rev_cholesky(B)) ** 2
    E = np.asarray(E, dtype=np.float64)
    return float(np.sum(E * E * rb[:, None] * ra[None, :]))


def corollary34_bound(A, B):
    """(1/4 sum_ij R_B,ii^2 R_A,jj^2, 1/4 tr A tr B) for the alphabet Z."""
    ra = np.diag(rev_cholesky(A)) ** 2
    rb = np.diag(rev_cholesky(B)) ** 2
    inner = 0.25 * float(np.sum(rb) * np.sum(ra))
    outer = 0.25 * float(np.trace(np.asarray(A, np.float64)) * np.trace(np.asarray(B, np.float64)))
    return inner, outer


def match_fraction(V1, V2) -> float:
    """Fraction of identical integer codes."""
    V1 = np.asarray(V1)
    V2 = np.asarray(V2)
    if V1.size == 0:
        return 1.0
    return float(np.mean(V1 == V2))
