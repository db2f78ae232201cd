"""Tolerances of the GPU parity tests, each derived from the arithmetic.

Factors.  The library computes L-hat = Cholesky(H^-1) with unit columns
("BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 3.2,
Algorithm 1; App. B) in double-float arithmetic, whose unit roundoff is at
most 2^-44 (a pair of fp32 words keeps 44 to 48 significant bits), and
rounds the result once to fp32.  First-order perturbation theory for the
Cholesky factor and the triangular inverse bounds the relative error of a
factor computed with backward error u by about cond(H) times u; rounding
errors of d-term dot products grow like sqrt(d) when they are independent.
So entry (i, j) of the GPU factor may differ from the exact one by

    ulp_fp32(L_ij) + 2^-44 * cond_1(H) * sqrt(d) * max |L|

(the first term: one rounding to fp32 plus the case where the double-float
value sits next to an fp32 rounding boundary).  The fp64 oracle's own error
(2^-53 instead of 2^-44) is inside this bound.  cond_1(H) is LAPACK's
estimate from the Cholesky factor (dpocon), which is within a small factor
of the true 1-norm condition number.

Distortion.  With identical codes, the GPU's Wq = fp32(s v) and the
oracle's Wq = s v (fp64) differ entrywise by at most 2^-24 |Wq|, so with
H = A (x) B, ||x||_H^2 = vec(x)^T H vec(x) <= lambda_max(A) lambda_max(B)
||x||_F^2 and lambda_max <= ||.||_1,

    |D_gpu - D_oracle| <= 2 sqrt(D_oracle) q + q^2,
    q = 2^-24 sqrt(||A||_1 ||B||_1) ||Wq||_F.

The parity bar adds the north-star's 1e-4 relative allowance for the few
codes (at most 0.01%) that may differ at near-ties.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import cho_factor
from scipy.linalg.lapack import dpocon

DF_UNIT = 2.0**-44
FP32_UNIT = 2.0**-24


def cond1(H) -> float:
    """LAPACK estimate of the 1-norm condition number of the SPD matrix H."""
    H = np.asarray(H, dtype=np.float64)
    anorm = float(np.abs(H).sum(axis=0).max())
    c, _ = cho_factor(H, lower=False, check_finite=False)
    rcond, info = dpocon(c, anorm)  # c holds the upper Cholesky factor (uplo = "U")
    assert info == 0
    return 1.0 / max(float(rcond), 1e-300)


def factor_tolerance(R, H) -> np.ndarray:
    """Entrywise bound on |L-hat_gpu - L-hat_exact| (R: the fp64 oracle factor)."""
    R = np.asarray(R, dtype=np.float64)
    d = R.shape[0]
    ulp = np.spacing(np.abs(R).astype(np.float32)).astype(np.float64)
    return ulp + DF_UNIT * cond1(H) * np.sqrt(d) * float(np.abs(R).max())


def check_factor(G, R, H) -> float:
    """Unit lower triangle, and every entry within factor_tolerance; returns the
    largest error as a fraction of its bound."""
    G = np.asarray(G)
    assert np.array_equal(np.triu(G, 1), np.zeros_like(G))
    assert np.all(np.diag(G) == 1.0)
    err = np.abs(G.astype(np.float64) - R)
    frac = float((err / factor_tolerance(R, H)).max()) if G.size else 0.0
    assert frac <= 1.0, frac
    return frac


def distortion_tolerance(d_ref: float, Wq_ref, A, B, rel: float = 1e-4) -> float:
    """Allowed |D_gpu - D_oracle| (see the module docstring)."""
    a1 = float(np.abs(np.asarray(A, np.float64)).sum(axis=0).max())
    b1 = float(np.abs(np.asarray(B, np.float64)).sum(axis=0).max())
    q = FP32_UNIT * np.sqrt(a1 * b1) * float(np.linalg.norm(np.asarray(Wq_ref, np.float64)))
    return rel * abs(d_ref) + 2.0 * np.sqrt(max(d_ref, 0.0)) * q + q * q
