"""Pins of the oracle's scale search, code packing and explicit alphabets
(App. D of "BaKron: Efficient Quantization with Kronecker-Factored
Hessians"; Sec. 3.1 for the alphabet)."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_row_scales_golden_cases():
    cases = json.load(open(os.path.join(GOLDEN, "row_scales.json")))["cases"]
    for c in cases:
        s, g = O.row_scales(np.array([c["row"]], dtype=np.float32), c["lo"], c["hi"], c["grid"])
        assert g[0] == c["chosen"], c["derivation"]
        assert s[0] == np.float32(c["scale"]), c["derivation"]


def test_no_search_is_absmax_over_hi():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((20, 33)).astype(np.float32)
    for lo, hi in ((-8, 7), (-3, 3), (-2, 1)):
        s, g = O.row_scales(W, lo, hi, 1)
        assert np.array_equal(s, (np.abs(W).max(axis=1) / np.float32(hi)).astype(np.float32))
        assert not g.any()


def test_equal_magnitude_rows_keep_the_full_scale():
    # every |W_ij| = c with c / hi exact in fp32: at f = 1 every entry maps
    # exactly onto +-hi, a zero error no other factor can beat (equals keep g = 0)
    for lo, hi, c in ((-3, 3, 0.75), (-8, 7, 1.75), (-2, 1, 0.5)):
        W = np.array([[c, -c, c, c], [-c] * 4], dtype=np.float32)
        s, g = O.row_scales(W, lo, hi, 25)
        assert not g.any()
        assert np.all(s == np.float32(c / hi))


def _exact_error(w, s, lo, hi):
    """Round-to-nearest squared error in exact rational arithmetic (decision:
    the fp32 quotient rounded half to even)."""
    tot = Fraction(0)
    for x in np.asarray(w, dtype=np.float32):
        v = int(np.clip(np.rint(np.float32(x) / np.float32(s)), lo, hi))
        d = Fraction(float(x)) - Fraction(float(np.float32(s))) * v
        tot += d * d
    return tot


def test_chosen_scale_minimizes_the_exact_error():
    rng = np.random.default_rng(7)
    W = (rng.standard_t(3, size=(12, 17)) * 0.3).astype(np.float32)
    grid = 9
    f = O.shrink_factors(grid)
    for lo, hi in ((-3, 3), (-4, 3)):
        s, g = O.row_scales(W, lo, hi, grid)
        for i, w in enumerate(W):
            s0 = np.float32(np.abs(w).max() / np.float32(hi))
            errs = [_exact_error(w, np.float32(s0 * f[k]), lo, hi) for k in range(grid)]
            best = min(errs)
            assert errs[g[i]] == best and all(e > best for e in errs[: g[i]])
            assert s[i] == np.float32(s0 * f[g[i]])


def test_shrink_factors_span_one_to_one_half():
    f = O.shrink_factors(11)
    assert f[0] == 1.0 and f[-1] == 0.5 and np.all(np.diff(f) < 0)
    assert O.shrink_factors(1).tolist() == [1.0]


def test_pack_golden_bytes_and_round_trip():
    cases = json.load(open(os.path.join(GOLDEN, "pack_codes.json")))["cases"]
    for c in cases:
        V = np.array(c["codes"])
        P = O.pack_codes(V, c["bits"])
        assert P.tolist() == c["bytes"], c["derivation"]
        assert np.array_equal(O.unpack_codes(P, V.shape[1], c["bits"]), V)
    rng = np.random.default_rng(1)
    for bits in (2, 4, 8):
        V = rng.integers(-(1 << (bits - 1)), 1 << (bits - 1), size=(5, 37))
        assert np.array_equal(O.unpack_codes(O.pack_codes(V, bits), 37, bits), V)
    with pytest.raises(ValueError):
        O.pack_codes(np.array([[8]]), 4)


def test_explicit_alphabet_is_clamped_rounding_for_diagonal_factors():
    # L-hat = I on both sides: every entry is rounded on its own (App. B eq. (2))
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((9, 13)) * 2.0).astype(np.float32)
    s = np.full(9, 0.5, dtype=np.float32)
    V, Wq, _ = O.bakron(W, LA=np.eye(13), LB=np.eye(9), scales=s, bits=(-3, 3))
    expect = np.clip(np.rint(W / np.float32(0.5)), -3, 3)
    assert np.array_equal(V, expect)
    assert O.alphabet_bounds((-3, 3)) == (-3, 3) and O.alphabet_bounds(4) == (-8, 7)
