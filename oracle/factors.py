"""Factor preparation, in float64 (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians":
  Sec. 3.1 defines Cholesky(H) as the lower-triangular L with L L^T = H and
  positive diagonal, and RevCholesky(H) as the lower-triangular L with
  L^T L = H and positive diagonal.
  Sec. 3.2, Algorithm 1 (and Algorithms 2, 3, 5, 6): L = Cholesky(H^-1), then
  every column is divided by its diagonal entry, so that L-hat is unit lower
  triangular.  App. B: this is done once, at the top level.
"""

from __future__ import annotations

import numpy as np


def normalized_inv_cholesky(H: np.ndarray) -> np.ndarray:
    """L-hat = Cholesky(H^-1) with each column divided by its diagonal entry.

    Written as the plain definition: invert H, factor the inverse with the
    library Cholesky routine, normalize the columns.  float64 throughout.
    """
    H = np.asarray(H, dtype=np.float64)
    Hinv = np.linalg.inv(H)
    Hinv = 0.5 * (Hinv + Hinv.T)  # exact symmetry for the factorization
    L = np.linalg.cholesky(Hinv)
    return L / np.diag(L)[None, :]


def rev_cholesky(H: np.ndarray) -> np.ndarray:
    """RevCholesky(H): the lower-triangular R with R^T R = H, positive diagonal.

    With J the reversal permutation, C = Cholesky(J H J) gives
    H = (J C J)(J C J)^T, and J C J is upper triangular, so R = (J C J)^T.
    """
    H = np.asarray(H, dtype=np.float64)
    C = np.linalg.cholesky(H[::-1, ::-1])
    return np.ascontiguousarray(C[::-1, ::-1].T)
