"""Seeded synthetic calibration samples for the Hessian-factor accumulation.

A layer's input activations a_t (n features) and backpropagated output-side
vectors b_t (m outputs), one sample per column, stored feature-major
(features x samples, row-major) as bfloat16 values: ``*_bits`` holds the
uint16 bit patterns the GPU reads, ``*_f32`` the same values as float32 for
the oracle.  Distributions follow the 4096 x 4096 workload's recipe: inputs
Student-t (nu = 4, heavy-tailed, as activations), outputs Gaussian with
AR(1) correlation rho = 0.9 along the output index.  Rounding float32 to
bfloat16 (to nearest, ties to even) is the input encoding, not part of the
method.
"""

from __future__ import annotations

import dataclasses

import numpy as np


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bfloat16 patterns of float32 values, rounded to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Samples:
    name: str
    n: int
    m: int
    N: int
    a_bits: np.ndarray  # uint16, n x N
    b_bits: np.ndarray  # uint16, m x N

    @property
    def a_f32(self) -> np.ndarray:
        return from_bf16_bits(self.a_bits)

    @property
    def b_f32(self) -> np.ndarray:
        return from_bf16_bits(self.b_bits)


def make_samples(n: int, m: int, N: int, seed: int = 0, scale: float = 1.0) -> Samples:
    """Student-t inputs and AR(1) Gaussian outputs, N samples each."""
    rng = np.random.default_rng(seed)
    a = scale * rng.standard_t(4.0, size=(n, N))
    z = rng.standard_normal((m, N))
    b = np.empty_like(z)
    if m:
        b[0] = z[0]
        c = np.sqrt(1.0 - 0.9 ** 2)
        for i in range(1, m):
            b[i] = 0.9 * b[i - 1] + c * z[i]
    return Samples(f"samples_{n}x{m}_N{N}_s{seed}", n, m, N, to_bf16_bits(a.astype(np.float32)),
                   to_bf16_bits(b.astype(np.float32)))


# Workloads: the input side of the 4096 x 4096 layer and of the 14336-wide
# layers, 65536 samples (32 sequences of 2048 tokens, one calibration slice).
SAMPLE_CONFIGS = {
    "g3": dict(n=4096, m=4096, N=65536, seed=5003),
    "g4": dict(n=14336, m=4096, N=16384, seed=5004),
}


def make_sample_config(key: str) -> Samples:
    return make_samples(**SAMPLE_CONFIGS[key])
