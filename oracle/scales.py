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

Groups and column scales (Sec. 3.1: scales "for each row and/or column";
App. D itself uses per-row scales, no groups).  The reading used: with a
group size g, row i holds one scale per run of g consecutive columns, each
chosen by the search above on that run alone (g >= n: one per row); column
scales t_j, where given, multiply in, and an entry's scale is the product
rounded once to fp32,
    sigma_ij = fp32(R[i, floor(j / g)] * t_j)  (sigma_ij = R[i, floor(j / g)]
without column scales); the alphabet of entry (i, j) is sigma_ij {lo .. hi}.

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


def row_scales(W, lo: int, hi: int, grid: int = 1, group=None):
    """Per-row scales (float32) and, per row, the index g chosen; with a
    ``group`` size, an (m, ceil(n / group)) array of per-run scales (and
    indices) instead."""
    if not (lo < 0 < hi):
        raise ValueError("the alphabet must contain negative and positive codes")
    W = np.asarray(W, dtype=np.float32)
    if group is not None:
        if group < 1:
            raise ValueError("group >= 1")
        m, n = W.shape
        ng = max(1, -(-n // group))
        S = np.empty((m, ng), dtype=np.float32)
        C = np.zeros((m, ng), dtype=np.int64)
        for k in range(ng):
            S[:, k], C[:, k] = row_scales(W[:, k * group:(k + 1) * group], lo, hi, grid)
        return S, C
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


def element_scales(R, n: int, group=None, col_scales=None) -> np.ndarray:
    """The m x n float32 scale of every entry: fp32(R[i, floor(j / g)] t_j).

    R: per-row scales (m,) (no groups) or per-run scales (m, ceil(n / g)).
    col_scales: n column scales t_j, or None (all ones, no rounding)."""
    R = np.asarray(R, dtype=np.float32)
    if R.ndim == 1:
        R = R[:, None]
    g = n if group is None else int(group)
    cols = np.arange(n) // g
    if R.shape[1] != max(1, -(-n // g)):
        raise ValueError("R must hold ceil(n / group) scales per row")
    S = R[:, cols]
    if col_scales is None:
        return np.ascontiguousarray(S)
    t = np.asarray(col_scales, dtype=np.float32)
    return (S.astype(np.float64) * t.astype(np.float64)[None, :]).astype(np.float32)


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
