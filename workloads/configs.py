"""The five benchmark workloads and small random problems, all seeded.

Every array is drawn in float64 with ``numpy.random.default_rng(seed)`` (PCG64)
and stored as float32: the float32 arrays are the canonical inputs, which the
oracle promotes to float64 and the CUDA path reads as they are.

A Gram factor is ``G = X X^T / N`` with one sample per column of ``X``; a
damped Gram factor adds ``damp * mean(diag(G)) * I``.  Seeds: W uses
``1000 + c``, the sample matrix behind A uses ``2000 + c``, the one behind B
``3000 + c`` and the spike directions ``4000 + c``, for workload number c.

Workloads (the shapes of the BaKron paper's Table 3, "BaKron: Efficient
Quantization with Kronecker-Factored Hessians", Section 6):

  c1  64 x 64       W ~ N(0,1); A = X X^T/512 + 0.01 I (X 64x512 Gaussian), B likewise;
                    alphabet Z (plain rounding), no scales.
  c2  1024 x 1024   W ~ N(0, 0.02^2); A, B damped Gaussian Grams (N = 4096, damp 1e-2);
                    4-bit alphabet {-8..7}, per-row absmax scales.
  c3  4096 x 4096   W ~ N(0, 0.02^2); A from N = 8192 Student-t (nu = 4) inputs,
                    B from N = 8192 Gaussian samples with AR(1) rho = 0.9 across the
                    outputs, both damped with 1e-2; 4-bit, per-row scales.
  c4  14336 x 4096  W ~ N(0, 0.02^2); A, B damped Gaussian Grams (N = 16384);
                    3-bit {-4..3}, per-row scales.
  c5  4096 x 14336  W ~ N(0, 0.02^2); A = I + U diag(99) U^T with U (14336 x 10)
                    orthonormal (ten eigenvalues 100, the rest 1); B damped Gaussian
                    Gram (N = 16384); 2-bit {-2..1}, per-row scales.

Per-row scales are ``max_j |W_ij| / (2^(bits-1) - 1)`` (the symmetric absmax
rule of the paper's Appendix D without its optional MSE shrink); for 2 bits
that is the plain absmax.
"""

from __future__ import annotations

import dataclasses
import hashlib
import os
from typing import Callable, Optional

import numpy as np


@dataclasses.dataclass
class Problem:
    """One quantization problem: quantize W (m x n) under the Hessian A (x) B."""

    name: str
    m: int
    n: int
    W: np.ndarray  # float32, m x n, row-major
    A: np.ndarray  # float32, n x n, symmetric positive definite
    B: np.ndarray  # float32, m x m, symmetric positive definite
    scales: Optional[np.ndarray]  # float32, m, or None (all ones)
    bits: int  # 0 = alphabet Z, else {-2^(bits-1) .. 2^(bits-1)-1}

    def digest(self) -> str:
        """SHA-256 over all arrays, to tag results with the exact inputs used."""
        h = hashlib.sha256()
        for arr in (self.W, self.A, self.B, self.scales):
            if arr is not None:
                h.update(np.ascontiguousarray(arr).tobytes())
        h.update(str(self.bits).encode())
        return h.hexdigest()[:16]


def _gram(X: np.ndarray, damp: float) -> np.ndarray:
    """X X^T / N (+ damp * mean(diag) * I), float64, symmetric."""
    N = X.shape[1]
    try:
        from scipy.linalg.blas import dsyrk

        G = dsyrk(1.0 / N, X)  # upper triangle of X X^T / N
        G = np.triu(G) + np.triu(G, 1).T
    except Exception:  # pragma: no cover - scipy is present on both machines
        G = (X @ X.T) / N
    if damp:
        G[np.diag_indices_from(G)] += damp * float(np.mean(np.diag(G)))
    return G


def _gaussian_gram(rng: np.random.Generator, d: int, N: int, damp: float) -> np.ndarray:
    return _gram(rng.standard_normal((d, N)), damp)


def _student_t_gram(rng: np.random.Generator, d: int, N: int, nu: float, damp: float) -> np.ndarray:
    return _gram(rng.standard_t(nu, size=(d, N)), damp)


def _ar1_gram(rng: np.random.Generator, d: int, N: int, rho: float, damp: float) -> np.ndarray:
    """Gram of N samples whose coordinates follow a stationary AR(1) chain."""
    Z = rng.standard_normal((d, N))
    Y = np.empty_like(Z)
    Y[0] = Z[0]
    c = np.sqrt(1.0 - rho * rho)
    for i in range(1, d):
        Y[i] = rho * Y[i - 1] + c * Z[i]
    return _gram(Y, damp)


def _spiked(rng: np.random.Generator, d: int, k: int, spike: float) -> np.ndarray:
    """I + U diag(spike - 1) U^T with U (d x k) orthonormal."""
    U, _ = np.linalg.qr(rng.standard_normal((d, k)))
    A = (spike - 1.0) * (U @ U.T)
    A[np.diag_indices_from(A)] += 1.0
    return 0.5 * (A + A.T)


def row_absmax_scales(W: np.ndarray, bits: int) -> np.ndarray:
    """Per-row scale max_j |W_ij| / (2^(bits-1) - 1), computed in float64, stored float32."""
    levels = (1 << (bits - 1)) - 1 if bits > 1 else 1
    s = np.max(np.abs(W.astype(np.float64)), axis=1) / levels
    s[s == 0] = 1.0
    return s.astype(np.float32)


def toeplitz_ar1(d: int, rho: float) -> np.ndarray:
    """The AR(1) covariance matrix rho^|i-j| (float64)."""
    idx = np.arange(d)
    return rho ** np.abs(idx[:, None] - idx[None, :]).astype(np.float64)


def _f32(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


def _c1() -> Problem:
    c, m, n = 1, 64, 64
    W = np.random.default_rng(1000 + c).standard_normal((m, n))
    A = _gram(np.random.default_rng(2000 + c).standard_normal((n, 512)), 0.0) + 0.01 * np.eye(n)
    B = _gram(np.random.default_rng(3000 + c).standard_normal((m, 512)), 0.0) + 0.01 * np.eye(m)
    return Problem("c1_64x64_Z", m, n, _f32(W), _f32(A), _f32(B), None, 0)


def _c2() -> Problem:
    c, m, n, bits = 2, 1024, 1024, 4
    W = _f32(0.02 * np.random.default_rng(1000 + c).standard_normal((m, n)))
    A = _gaussian_gram(np.random.default_rng(2000 + c), n, 4096, 1e-2)
    B = _gaussian_gram(np.random.default_rng(3000 + c), m, 4096, 1e-2)
    return Problem("c2_1024x1024_int4", m, n, W, _f32(A), _f32(B), row_absmax_scales(W, bits), bits)


def _c3() -> Problem:
    c, m, n, bits = 3, 4096, 4096, 4
    W = _f32(0.02 * np.random.default_rng(1000 + c).standard_normal((m, n)))
    A = _student_t_gram(np.random.default_rng(2000 + c), n, 8192, 4.0, 1e-2)
    B = _ar1_gram(np.random.default_rng(3000 + c), m, 8192, 0.9, 1e-2)
    return Problem("c3_4096x4096_int4", m, n, W, _f32(A), _f32(B), row_absmax_scales(W, bits), bits)


def _c4() -> Problem:
    c, m, n, bits = 4, 14336, 4096, 3
    W = _f32(0.02 * np.random.default_rng(1000 + c).standard_normal((m, n)))
    A = _gaussian_gram(np.random.default_rng(2000 + c), n, 16384, 1e-2)
    B = _gaussian_gram(np.random.default_rng(3000 + c), m, 16384, 1e-2)
    return Problem("c4_14336x4096_int3", m, n, W, _f32(A), _f32(B), row_absmax_scales(W, bits), bits)


def _c5() -> Problem:
    c, m, n, bits = 5, 4096, 14336, 2
    W = _f32(0.02 * np.random.default_rng(1000 + c).standard_normal((m, n)))
    A = _spiked(np.random.default_rng(4000 + c), n, 10, 100.0)
    B = _gaussian_gram(np.random.default_rng(3000 + c), m, 16384, 1e-2)
    return Problem("c5_4096x14336_int2", m, n, W, _f32(A), _f32(B), row_absmax_scales(W, bits), bits)


CONFIGS: dict[str, Callable[[], Problem]] = {
    "c1": _c1,
    "c2": _c2,
    "c3": _c3,
    "c4": _c4,
    "c5": _c5,
}


def make_config(key: str) -> Problem:
    """Build workload ``key`` ('c1'..'c5').

    If the environment variable BAKRON_INPUT_CACHE names a directory, the
    float32 arrays are cached there as .npz files keyed by the workload name.
    """
    cache = os.environ.get("BAKRON_INPUT_CACHE")
    if cache:
        path = os.path.join(cache, f"{key}.npz")
        if os.path.exists(path):
            z = np.load(path)
            s = z["scales"] if z["scales"].size else None
            return Problem(str(z["name"]), int(z["m"]), int(z["n"]), z["W"], z["A"], z["B"], s, int(z["bits"]))
    p = CONFIGS[key]()
    if cache:
        os.makedirs(cache, exist_ok=True)
        np.savez(
            os.path.join(cache, f"{key}.npz"),
            name=p.name, m=p.m, n=p.n, W=p.W, A=p.A, B=p.B,
            scales=p.scales if p.scales is not None else np.zeros(0, np.float32), bits=p.bits,
        )
    return p


def random_problem(
    m: int,
    n: int,
    bits: int = 4,
    seed: int = 0,
    kind: str = "gram",
    w_std: float = 1.0,
    samples: Optional[int] = None,
) -> Problem:
    """A small seeded problem of any shape.

    kind:
      'gram'      damped Gaussian Gram factors (N = max(2d, 8) samples, damp 1e-2)
      'identity_b'  A a damped Gram, B = I (the one-sided, row-wise case)
      'diagonal'  A, B positive diagonal matrices
      'ar1'       A = I, B = the AR(1) covariance rho^|i-j| with rho = 0.9
    W ~ N(0, w_std^2); with bits > 0 the rows get absmax scales.
    """
    rng = np.random.default_rng(seed)
    W = w_std * rng.standard_normal((m, n))
    if kind == "gram":
        A = _gaussian_gram(rng, n, samples or max(2 * n, 8), 1e-2)
        B = _gaussian_gram(rng, m, samples or max(2 * m, 8), 1e-2)
    elif kind == "identity_b":
        A = _gaussian_gram(rng, n, samples or max(2 * n, 8), 1e-2)
        B = np.eye(m)
    elif kind == "diagonal":
        A = np.diag(rng.uniform(0.5, 2.0, n))
        B = np.diag(rng.uniform(0.5, 2.0, m))
    elif kind == "ar1":
        A = np.eye(n)
        B = toeplitz_ar1(m, 0.9)
    else:
        raise ValueError(f"unknown kind {kind!r}")
    W32 = _f32(W)
    scales = row_absmax_scales(W32, bits) if bits > 0 else None
    return Problem(f"rand_{kind}_{m}x{n}_b{bits}_s{seed}", m, n, W32, _f32(A), _f32(B), scales, bits)
