"""Divide-and-conquer solvers (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians":
  Sec. 3.4, Algorithm 5 (BaKron-recursive): if m < n, solve the left half of
  the columns, add L_B (V - W)_left (L_A[right, left])^T to the right half,
  solve the right half; otherwise split the rows the same way with
  L_B[bottom, top] (V - W)_top L_A^T.  Base case: one entry.
  Sec. 3.5, Algorithm 6 (BaKron): the same over ranges k:l of anti-diagonals:
  solve k:mid, add antidiag_{mid:l}(L_B (V - antidiag_{k:mid} W) L_A^T),
  solve mid:l.  Base case: round one anti-diagonal.
  App. B conventions: the factors are prepared once at the top level and
  the children get sub-blocks of them; children work in place on one shared
  workspace, which keeps on a finished set the values its entries were
  rounded at, so that V - W there is the error matrix E.  Midpoints are
  floor((k+l)/2) (App. C: n1 = floor(n/2)); Theorem 3.2 makes the output
  independent of the split.

The errors are kept in a separate array E at rounding time, which is the
same as "V - W on the finished set" in the paper's convention.
"""

from __future__ import annotations

import sys

import numpy as np

from .antidiag import antidiagonal_indices
from .quantizer import quantize, scale_at, scale_grid


def _scales32(scales):
    return None if scales is None else np.asarray(scales, dtype=np.float32)


def bakron_recursive(W, LA, LB, scales, bits: int, leaf: int = 64):
    """Algorithm 5.  Blocks of at most ``leaf`` x ``leaf`` entries are solved by
    Algorithm 3 restricted to the block (with the diagonal blocks of the
    factors), which Theorem 3.2 makes equal to recursing down to single
    entries; ``leaf=1`` recurses to single entries as the algorithm is printed.

    Returns (V int64, Wq float64, E float64), all m x n.
    """
    Wk = np.array(W, dtype=np.float64)
    LA = np.asarray(LA, dtype=np.float64)
    LB = np.asarray(LB, dtype=np.float64)
    s = _scales32(scales)
    m, n = Wk.shape
    V = np.zeros((m, n), dtype=np.int64)
    E = np.zeros((m, n))

    def leaf_block(r0, r1, c0, c1):
        lb = LB[r0:r1, r0:r1]
        la = LA[c0:c1, c0:c1]
        blk = Wk[r0:r1, c0:c1]
        mm, nn = r1 - r0, c1 - c0
        for k in range(mm + nn - 1):
            rows, cols = antidiagonal_indices(mm, nn, k)
            v, d = quantize(blk[rows, cols], scale_at(s, r0 + rows, c0 + cols), bits)
            V[r0 + rows, c0 + cols] = v
            E[r0 + rows, c0 + cols] = d
            blk += (lb[:, rows] * d[None, :]) @ la[:, cols].T

    def solve(r0, r1, c0, c1):
        mm, nn = r1 - r0, c1 - c0
        if mm == 1 and nn == 1:
            v, d = quantize(Wk[r0, c0], scale_at(s, r0, c0), bits)
            V[r0, c0] = v
            E[r0, c0] = d
        elif leaf > 1 and mm <= leaf and nn <= leaf:
            leaf_block(r0, r1, c0, c1)
        elif mm < nn:
            h = nn // 2
            solve(r0, r1, c0, c0 + h)
            Wk[r0:r1, c0 + h:c1] += (LB[r0:r1, r0:r1] @ E[r0:r1, c0:c0 + h]) @ LA[c0 + h:c1, c0:c0 + h].T
            solve(r0, r1, c0 + h, c1)
        else:
            h = mm // 2
            solve(r0, r0 + h, c0, c1)
            Wk[r0 + h:r1, c0:c1] += (LB[r0 + h:r1, r0:r0 + h] @ E[r0:r0 + h, c0:c1]) @ LA[c0:c1, c0:c1].T
            solve(r0 + h, r1, c0, c1)

    old = sys.getrecursionlimit()
    sys.setrecursionlimit(max(old, 10000))
    try:
        solve(0, m, 0, n)
    finally:
        sys.setrecursionlimit(old)
    Wq = scale_grid(s, m, n) * V
    return V, Wq, E


def bakron_alg6(W, LA, LB, scales, bits: int):
    """Algorithm 6 over the full matrix (dense masked products; tiny inputs).

    Returns (V, Wq, E).
    """
    Wk = np.array(W, dtype=np.float64)
    LA = np.asarray(LA, dtype=np.float64)
    LB = np.asarray(LB, dtype=np.float64)
    s = _scales32(scales)
    m, n = Wk.shape
    V = np.zeros((m, n), dtype=np.int64)
    E = np.zeros((m, n))
    kidx = np.add.outer(np.arange(m), np.arange(n))

    def solve(k, l):
        if l == k + 1:
            rows, cols = antidiagonal_indices(m, n, k)
            v, d = quantize(Wk[rows, cols], scale_at(s, rows, cols), bits)
            V[rows, cols] = v
            E[rows, cols] = d
            return
        mid = (k + l) // 2
        solve(k, mid)
        Eband = np.where((kidx >= k) & (kidx < mid), E, 0.0)
        P = LB @ Eband @ LA.T
        Wk[...] += np.where((kidx >= mid) & (kidx < l), P, 0.0)
        solve(mid, l)

    solve(0, m + n - 1)
    Wq = scale_grid(s, m, n) * V
    return V, Wq, E
