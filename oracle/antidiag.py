"""Anti-diagonal solvers (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians":
  Sec. 3.1: anti-diagonal k holds the entries (i, j) with i + j = k; in
  0-based indices k runs over 0 .. m+n-2.
  App. B, eq. (2): the order-free definition of the result,
      W~_k = Pi_{I_k}( W0 + L_B (sum_{l<k} E_l) L_A^T ),
      V_k = round(W~_k),  E_k = V_k - W~_k.
  Sec. 3.3, Algorithm 3 (BaKron-antidiagonal): for every anti-diagonal k,
      D = antidiag_k(W), V = round(D), Delta = V - D, W += L_B Delta L_A^T.

Both take the already normalized factors L-hat_A (n x n) and L-hat_B (m x m).
"""

from __future__ import annotations

import numpy as np

from .quantizer import quantize, scale_at


def antidiagonal_indices(m: int, n: int, k: int):
    """Row and column indices of anti-diagonal k (0-based), rows ascending."""
    i0 = max(0, k - (n - 1))
    i1 = min(m - 1, k)
    rows = np.arange(i0, i1 + 1)
    return rows, k - rows




def bakron_definition(W, LA, LB, scales, bits: int):
    """App. B eq. (2), evaluated literally: one full L_B E L_A^T per anti-diagonal.

    O(mn(m+n)) per anti-diagonal -- for tiny inputs only.  Returns (V, Wq, E).
    """
    W0 = np.asarray(W, dtype=np.float64)
    LA = np.asarray(LA, dtype=np.float64)
    LB = np.asarray(LB, dtype=np.float64)
    m, n = W0.shape
    V = np.zeros((m, n), dtype=np.int64)
    E = np.zeros((m, n))
    for k in range(m + n - 1):
        rows, cols = antidiagonal_indices(m, n, k)
        Wt = W0 + LB @ E @ LA.T  # E is zero on anti-diagonals >= k
        v, e = quantize(Wt[rows, cols], scale_at(scales, rows, cols), bits)
        V[rows, cols] = v
        E[rows, cols] = e
    Wq = W0 + LB @ E @ LA.T
    return V, Wq, E


def bakron_antidiagonal(W, LA, LB, scales, bits: int):
    """Algorithm 3: round one anti-diagonal, then one batched rank-d update.

    Returns (V, Wq, E); the final workspace is Wq (the unit diagonal of the
    factors turns every rounded entry into its quantized value).
    """
    Wk = np.array(W, dtype=np.float64)
    LA = np.asarray(LA, dtype=np.float64)
    LB = np.asarray(LB, dtype=np.float64)
    m, n = Wk.shape
    V = np.zeros((m, n), dtype=np.int64)
    E = np.zeros((m, n))
    for k in range(m + n - 1):
        rows, cols = antidiagonal_indices(m, n, k)
        v, delta = quantize(Wk[rows, cols], scale_at(scales, rows, cols), bits)
        V[rows, cols] = v
        E[rows, cols] = delta
        # L_B Delta L_A^T with Delta supported on the anti-diagonal
        Wk += (LB[:, rows] * delta[None, :]) @ LA[:, cols].T
    return V, Wk, E
