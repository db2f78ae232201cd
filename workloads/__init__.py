"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This package draws the numbers that both sides of a parity check receive: the
weight matrix W, the two positive-definite Kronecker factors A (n x n, input
side) and B (m x m, output side) and the per-row scales.  It contains none of
the quantization method's arithmetic, and it imports neither the oracle nor
the CUDA package.
"""

from .configs import (  # noqa: F401
    CONFIGS,
    Problem,
    make_config,
    random_problem,
    row_absmax_scales,
    toeplitz_ar1,
)
