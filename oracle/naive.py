"""Brute-force solvers on the vectorized weights (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians":
  Sec. 3.1: vec(W) is the column-major flattening, so entry (i, j) of an
  m x n matrix is coordinate i + m*j, and (A (x) B) vec(W) = vec(B W A^T)
  (Proposition 3.1).
  Sec. 3.2, Algorithm 1: GPTQ on one vector: L = Cholesky(H^-1), columns
  normalized by their diagonal; for i = 1..n: v = round(w_i),
  Delta = v - w_i, w += Delta * L_i.
  Sec. 3.2: BaKron-naive is Algorithm 1 applied to w = vec(W), H = A (x) B.
  Sec. 3.2 also relates GPTQ to Babai's nearest-plane algorithm for the
  lattice with basis M, M^T M = H; ``babai_nearest_plane`` is that second,
  independent formulation (successive rounding in the triangular basis
  R = RevCholesky(H)), used only to pin the naive solver.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from .factors import normalized_inv_cholesky, rev_cholesky
from .quantizer import quantize


def _vec_scales(scales: Optional[np.ndarray], m: int, n: int) -> Optional[np.ndarray]:
    """Scale of every coordinate of vec(W): coordinate t is entry (t mod m,
    t div m).  ``scales``: one per row (m,) or one per entry (m, n)."""
    if scales is None:
        return None
    s = np.asarray(scales, dtype=np.float32)
    return np.tile(s, n) if s.ndim == 1 else s.flatten(order="F")


def gptq_vector(w: np.ndarray, Lhat: np.ndarray, s: Optional[np.ndarray], bits: int):
    """Algorithm 1 on one vector with a given normalized factor.

    Returns (codes, errors at rounding time, final w).  ``s`` holds one float32
    scale per coordinate (or None).
    """
    w = np.array(w, dtype=np.float64)
    N = w.shape[0]
    codes = np.zeros(N, dtype=np.int64)
    errs = np.zeros(N, dtype=np.float64)
    for t in range(N):
        v, e = quantize(w[t], None if s is None else s[t], bits)
        codes[t] = v
        errs[t] = e
        w += e * Lhat[:, t]
    return codes, errs, w


def bakron_naive(W, A, B, scales, bits: int):
    """BaKron-naive: Algorithm 1 on vec(W) with the explicit H = A (x) B.

    Returns (V int64 m x n, Wq float64 m x n, E float64 m x n).  Only for
    small m*n: it forms the (mn x mn) Kronecker product.
    """
    W = np.asarray(W, dtype=np.float64)
    m, n = W.shape
    H = np.kron(np.asarray(A, dtype=np.float64), np.asarray(B, dtype=np.float64))
    Lhat = normalized_inv_cholesky(H)
    codes, errs, w = gptq_vector(W.flatten(order="F"), Lhat, _vec_scales(scales, m, n), bits)
    V = codes.reshape((m, n), order="F")
    E = errs.reshape((m, n), order="F")
    Wq = w.reshape((m, n), order="F")
    return V, Wq, E


def babai_nearest_plane(W, A, B, scales, bits: int):
    """Successive rounding in the basis R = RevCholesky(A (x) B).

    Minimizing ||R (v - w)||_2 coordinate by coordinate: since R is lower
    triangular, coordinate t of R (v - w) involves v_1..v_t only, and it is
    made as small as the alphabet allows by
        v_t = quantize( w_t - sum_{j<t} R_tj (v_j - w_j) / R_tt ).
    Returns (V, E) with E = v - (rounded-at value), m x n.
    """
    W = np.asarray(W, dtype=np.float64)
    m, n = W.shape
    H = np.kron(np.asarray(A, dtype=np.float64), np.asarray(B, dtype=np.float64))
    R = rev_cholesky(H)
    w = W.flatten(order="F")
    s = _vec_scales(scales, m, n)
    N = w.shape[0]
    diff = np.zeros(N)  # v_j - w_j for the coordinates decided so far
    codes = np.zeros(N, dtype=np.int64)
    errs = np.zeros(N)
    for t in range(N):
        target = w[t] - np.dot(R[t, :t], diff[:t]) / R[t, t]
        v, e = quantize(target, None if s is None else s[t], bits)
        codes[t] = v
        errs[t] = e
        sv = (1.0 if s is None else np.float64(s[t])) * v
        diff[t] = sv - w[t]
    return codes.reshape((m, n), order="F"), errs.reshape((m, n), order="F")


def gptq_rows(W, A, scales, bits: int):
    """Row-wise GPTQ: Algorithm 1 with H = A run on every row of W.

    This is the one-sided case B = I (Sec. 1: GPTQ's Hessian is X X^T (x) I).
    Returns (V, Wq, E).
    """
    W = np.asarray(W, dtype=np.float64)
    m, n = W.shape
    Lhat = normalized_inv_cholesky(A)
    V = np.zeros((m, n), dtype=np.int64)
    E = np.zeros((m, n))
    Wq = np.zeros((m, n))
    for i in range(m):
        if scales is None:
            s = None
        else:
            sc = np.asarray(scales, dtype=np.float32)
            s = np.full(n, sc[i], dtype=np.float32) if sc.ndim == 1 else sc[i]
        V[i], E[i], Wq[i] = gptq_vector(W[i], Lhat, s, bits)
    return V, Wq, E
