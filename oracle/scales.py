"""Per-row scale choice and packed codes (oracle; test infrastructure only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians", App. D:
scales are chosen per output feature (per row of W): the row's largest
absolute value divided by l for the alphabet {-l .. l}, then optionally
shrunk "by up to a factor of 2 based on an MSE search".  The pages do not
spell the search out; the reading used here is the plain one:

* base scale  s0 = fp32(max_j |W_ij| / hi)  (one correctly rounded fp32
  division; hi = l for the symmetric alphabet, the largest code otherwise);
* shrink factors f_g = fp32(1 - g / (2 (G - 1))), g = 0 .. G-1 (G >= 2),
  from 1 down to 1/2; candidate scale s_g = fp32(s0 * f_g);
* the row's round-to-nearest error for s_g is sum_j (W_ij - s_g v_ij)^2 with
  v_ij = clamp(round_half_even(fp32(W_ij) / s_g), lo, hi) (the decision in
  fp32, as everywhere in the solve);
* the chosen scale is the s_g of least error, the smallest g among equals.

G = 1 means no search (s0).  A row of zeros gets scale 1.

Packed codes: each code v in {lo .. hi}, lo >= -2^(b-1), hi < 2^(b-1), is
stored as its b-bit two's complement, b in {2, 4, 8}; code j of a row sits
in byte floor(j b / 8) at bit offset (j b) mod 8 (little-endian within the
byte); each row starts at a byte boundary, rows ceil(n b / 8) bytes long.
"""

from __future__ import annotations

import numpy as np


def shrink_factors(grid: int) -> np.ndarray:
    """The fp32 shrink factors f_0 .. f_{G-1}."""
    if grid < 1:
        raise ValueError("grid >= 1")
    if grid == 1:
        return np.ones(1, dtype=np.float32)
    g = np.arange(grid, dtype=np.float64)
    return (1.0 - g / (2.0 * (grid - 1))).astype(np.float32)


def row_error(w, s, lo: int, hi: int) -> float:
    """Round-to-nearest squared error of one row for the fp32 scale s, in fp64
    (s v is exact in fp64: 24-bit scale times an integer below 2^15)."""
    w32 = np.asarray(w, dtype=np.float32)
    s32 = np.float32(s)
    v = np.clip(np.rint((w32 / s32).astype(np.float32)), lo, hi)
    e = w32.astype(np.float64) - np.float64(s32) * v.astype(np.float64)
    return float(np.dot(e, e))


def row_scales(W, lo: int, hi: int, grid: int = 1):
    """Per-row scales (float32) and, per row, the index g chosen."""
    if not (lo < 0 < hi):
        raise ValueError("the alphabet must contain negative and positive codes")
    W = np.asarray(W, dtype=np.float32)
    f = shrink_factors(grid)
    scales = np.empty(W.shape[0], dtype=np.float32)
    chosen = np.zeros(W.shape[0], dtype=np.int64)
    for i, w in enumerate(W):
        amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
        if amax == 0:
            scales[i] = 1.0
            continue
        s0 = np.float32(amax / np.float32(hi))
        best, best_err = 0, None
        for g in range(grid):
            s = np.float32(s0 * f[g])
            err = row_error(w, s, lo, hi)
            if best_err is None or err < best_err:
                best, best_err = g, err
        scales[i] = np.float32(s0 * f[best])
        chosen[i] = best
    return scales, chosen


def pack_codes(V, bits: int) -> np.ndarray:
    """m x ceil(n bits / 8) uint8 array of the b-bit two's complement codes."""
    if bits not in (2, 4, 8):
        raise ValueError("bits in {2, 4, 8}")
    V = np.asarray(V, dtype=np.int64)
    m, n = V.shape
    if V.size and (V.min() < -(1 << (bits - 1)) or V.max() >= (1 << (bits - 1))):
        raise ValueError("codes outside the b-bit range")
    per = 8 // bits
    rowbytes = (n * bits + 7) // 8
    out = np.zeros((m, rowbytes), dtype=np.uint8)
    mask = (1 << bits) - 1
    for j in range(n):
        out[:, j // per] |= ((V[:, j] & mask) << ((j % per) * bits)).astype(np.uint8)
    return out


def unpack_codes(P, n: int, bits: int) -> np.ndarray:
    """Inverse of pack_codes (sign-extended int64 codes)."""
    P = np.asarray(P, dtype=np.uint8)
    per = 8 // bits
    mask = (1 << bits) - 1
    V = np.zeros((P.shape[0], n), dtype=np.int64)
    for j in range(n):
        u = (P[:, j // per].astype(np.int64) >> ((j % per) * bits)) & mask
        V[:, j] = np.where(u >= (1 << (bits - 1)), u - (1 << bits), u)
    return V
