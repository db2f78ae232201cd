"""The scalar base quantizer (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 3.1:
with b+1 bits the alphabet is {-2^b, ..., 2^b - 1}, mapped to the weights'
range by per-row scale factors, and "round" is replaced by the map to the
closest alphabet element.  With ``bits`` = b+1 the alphabet here is
{-2^(bits-1) .. 2^(bits-1) - 1}; ``bits`` = 0 means the unbounded alphabet Z
(plain rounding, scale 1).  For a contiguous integer alphabet the closest
element of s*{lo..hi} to x is s * clamp(round(x / s), lo, hi).

Ties: App. B fixes "a rule for breaking rounding ties" without naming it; the
rule used is round half to even.

The decision is taken in float32 (the paper's implementation precision,
Sec. 6): x is converted to float32, divided by the float32 scale in one
correctly rounded float32 division, then rounded half to even.
"""

from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def alphabet_bounds(bits) -> Optional[Tuple[int, int]]:
    """(lo, hi) of the alphabet for ``bits`` > 0, or None for Z.

    ``bits`` may also be an explicit integer alphabet (lo, hi), lo < hi: the
    symmetric {-l .. l} of App. D is (-l, l)."""
    if isinstance(bits, tuple):
        lo, hi = int(bits[0]), int(bits[1])
        if not lo < hi:
            raise ValueError("an explicit alphabet needs lo < hi")
        return lo, hi
    if bits == 0:
        return None
    if bits < 2:
        raise ValueError("bits must be 0 (alphabet Z) or >= 2")
    half = 1 << (bits - 1)
    return -half, half - 1


def quantize(x, s, bits):
    """Integer codes v and float64 errors e = s*v - x for values x (float64).

    ``s`` is a float32 scale broadcastable to x, or None for scale 1.
    """
    x = np.asarray(x, dtype=np.float64)
    x32 = x.astype(np.float32)
    if s is None:
        y = x32
        s64 = np.float64(1.0)
    else:
        s32 = np.asarray(s, dtype=np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            y = (x32 / s32).astype(np.float32)
        s64 = s32.astype(np.float64)
    v = np.rint(y)
    b = alphabet_bounds(bits)
    if b is not None:
        v = np.clip(v, b[0], b[1])
    v = v.astype(np.int64)
    e = s64 * v.astype(np.float64) - x
    return v, e


def scale_at(scales, rows, cols):
    """The float32 scales of entries (rows[k], cols[k]): ``scales`` is None
    (scale 1), one scale per row (shape (m,)), or one per entry (shape
    (m, n); see oracle.scales.element_scales for row, group and column
    scales)."""
    if scales is None:
        return None
    s = np.asarray(scales, dtype=np.float32)
    return s[rows] if s.ndim == 1 else s[rows, cols]


def scale_grid(scales, m: int, n: int):
    """The m x n float64 matrix of every entry's scale (1 for None)."""
    if scales is None:
        return np.ones((m, n))
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return np.broadcast_to(s[:, None] if s.ndim == 1 else s, (m, n))

