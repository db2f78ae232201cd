"""One entry point over the oracle's solvers (test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 3:
every solver takes W, the positive-definite factors A (n x n) and B (m x m),
prepares L-hat_A, L-hat_B once (Algorithm 1 prologue, App. B) and returns
the quantized matrix.  Theorem 3.2 makes all of them return the same V.
"""

from __future__ import annotations

import numpy as np

from .antidiag import bakron_antidiagonal, bakron_definition
from .factors import normalized_inv_cholesky
from .naive import bakron_naive
from .recursive import bakron_alg6, bakron_recursive


def factors_of(A, B):
    """(L-hat_A, L-hat_B) in float64 from the (float32) inputs promoted to float64."""
    return (
        normalized_inv_cholesky(np.asarray(A, dtype=np.float64)),
        normalized_inv_cholesky(np.asarray(B, dtype=np.float64)),
    )


def bakron(W, A=None, B=None, scales=None, bits=0, LA=None, LB=None, method="recursive", leaf=64):
    """Quantize W.  Give either A and B, or the normalized factors LA and LB.

    method: 'recursive' (Alg. 5, default), 'alg6', 'antidiagonal' (Alg. 3),
    'definition' (eq. (2)) or 'naive' (Alg. 1 on vec(W); needs A and B).
    Returns (V int64, Wq float64, E float64).
    """
    if method == "naive":
        return bakron_naive(W, A, B, scales, bits)
    if LA is None or LB is None:
        LA, LB = factors_of(A, B)
    if method == "recursive":
        return bakron_recursive(W, LA, LB, scales, bits, leaf=leaf)
    if method == "alg6":
        return bakron_alg6(W, LA, LB, scales, bits)
    if method == "antidiagonal":
        return bakron_antidiagonal(W, LA, LB, scales, bits)
    if method == "definition":
        return bakron_definition(W, LA, LB, scales, bits)
    raise ValueError(f"unknown method {method!r}")
