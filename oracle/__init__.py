"""fp64 CPU oracle for the BaKron solver -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The CUDA library never calls
into it, and it shares no code with the CUDA library: the two meet only in the
seeded input generators of the separate ``workloads`` package.

Source: "BaKron: Efficient Quantization with Kronecker-Factored Hessians"
(arXiv 2608.06291).  Every function names the section, algorithm or equation
it follows.

What is here, and what pins it (the pins live in ``tests/test_oracle_*.py``):

  factors.normalized_inv_cholesky   Sec. 3.2 Alg. 1 prologue.  Pinned by the
      closed form of the AR(1) covariance (L-hat = I - rho * subdiagonal),
      a hand-solved 2x2 case, and L-hat L-hat^T scaled = H^-1.
  factors.rev_cholesky             Sec. 3.1 definition.  Pinned by its
      defining properties (lower, positive diagonal, R^T R = H).
  quantizer.quantize               Sec. 3.1 alphabet.  Pinned by round-half-
      even golden values and clamping cases.
  naive.bakron_naive                Sec. 3.2 Alg. 1 applied to vec(W) with the
      explicit Kronecker product A (x) B.  Pinned against an independent
      Babai nearest-plane solver (successive rounding in the triangular
      basis RevCholesky(A (x) B)), and against round-to-nearest when A, B are
      diagonal.
  naive.gptq_rows                   Sec. 3.2 Alg. 1 run on every row (H = A).
      Used as the B = I pin of the two-sided solvers.
  antidiag.bakron_definition        App. B eq. (2), the order-free definition.
  antidiag.bakron_antidiagonal      Sec. 3.3 Alg. 3.
  recursive.bakron_recursive        Sec. 3.4 Alg. 5 (optionally with an Alg. 3
      leaf on small blocks, equal by Theorem 3.2).
  recursive.bakron_alg6             Sec. 3.5 Alg. 6.
      All four are pinned against the naive solver (Theorem 3.2: identical
      outputs), against the B = I and diagonal special cases, against a
      first-order error-feedback quantizer when A = I and B is AR(1), and by
      the exact identities of ``metrics``.
  metrics.*                         distortion tr(A (Wq-W)^T B (Wq-W)) and the
      two exact identities Wq - W = L_B E L_A^T and
      distortion = sum_ij E_ij^2 R_B,ii^2 R_A,jj^2, and Corollary 3.4's bound.
  quantizer.alphabet_bounds         also explicit alphabets (lo, hi), e.g. the
      symmetric {-l .. l} of App. D.  Pinned by clamped round-to-nearest
      when A and B are diagonal.
  scales.row_scales                 App. D scale choice (absmax / l, MSE
      shrink search up to 2x).  Pinned by hand-worked rows (tests/golden/
      row_scales.json), rows of equal magnitudes (zero error at the full
      scale) and the no-search case.
  scales.pack_codes / unpack_codes  b-bit two's complement packing.  Pinned
      by hand-packed bytes (tests/golden/pack_codes.json) and round trips.
  hessian.weighted_gram / kfac_factors / shampoo_factors / damp
      Kronecker factors from samples (Sec. 4.2, App. A.2, App. D damping).
      Pinned by hand-worked values (tests/golden/hessian.json), closed forms
      (orthogonal rows, single samples, a fixed output side), and the
      Van Loan-Pitsianis rearrangement of the explicit Kronecker sum: one
      Shampoo step is R(H) applied to the identity, many converge to the top
      singular pair.
  scales.element_scales             one scale per entry from per-row or
      per-run (group) scales and optional column scales (Sec. 3.1).  Pinned
      by hand-worked matrices; every solver accepts an m x n scale matrix,
      pinned by the naive solve on vec(W), per-entry rounding for diagonal
      factors, and power-of-two column scales as a change of variables
      (W D^-1, D A D) with identical codes.

No function here is "parity unpinned".

Rounding decisions are taken in float32 (the precision the paper's own
implementation uses, Sec. 6): the value to be rounded is computed in float64,
converted to float32, divided by the float32 row scale with one correctly
rounded float32 division and rounded half to even.  The error E = s*v - x is
then formed in float64 from the float64 value x.
"""

from .factors import normalized_inv_cholesky, rev_cholesky  # noqa: F401
from .quantizer import alphabet_bounds, quantize  # noqa: F401
from .hessian import damp, kfac_factors, shampoo_factors, squared_norms, weighted_gram  # noqa: F401
from .scales import element_scales, pack_codes, row_error, row_scales, shrink_factors, unpack_codes  # noqa: F401
from .naive import bakron_naive, babai_nearest_plane, gptq_rows  # noqa: F401
from .antidiag import bakron_antidiagonal, bakron_definition  # noqa: F401
from .recursive import bakron_alg6, bakron_recursive  # noqa: F401
from .metrics import (  # noqa: F401
    corollary34_bound,
    distortion,
    distortion_from_errors,
    errors_from_output,
    match_fraction,
)
from .api import bakron, factors_of  # noqa: F401
