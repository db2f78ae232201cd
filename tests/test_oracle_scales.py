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


# ------------------------------------------- groups and column scales (Sec. 3.1)

ENTRY_SOLVERS = ["definition", "antidiagonal", "alg6", "recursive1", "recursive64"]


def _entry_solve(W, LA, LB, S, bits, method):
    if method.startswith("recursive"):
        return O.bakron(W, LA=LA, LB=LB, scales=S, bits=bits, method="recursive", leaf=int(method[9:]))
    return O.bakron(W, LA=LA, LB=LB, scales=S, bits=bits, method=method)


def test_element_scales_hand_worked():
    # R: 2 rows x 2 runs of g = 3 over n = 5 columns; t: column scales.
    R = np.array([[2.0, 0.5], [1.0, 3.0]], dtype=np.float32)
    t = np.array([1.0, 0.5, 4.0, 1.0, 0.25], dtype=np.float32)
    expect = np.array([[2.0, 1.0, 8.0, 0.5, 0.125], [1.0, 0.5, 4.0, 3.0, 0.75]], dtype=np.float32)
    assert np.array_equal(O.element_scales(R, 5, group=3, col_scales=t), expect)
    assert np.array_equal(O.element_scales(R, 5, group=3), np.array([[2, 2, 2, 0.5, 0.5], [1, 1, 1, 3, 3]], np.float32))
    # the product is rounded once to fp32: (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 rounds (half to even) to 1 + 2^-11
    a = np.float32(1 + 2.0 ** -12)
    assert O.element_scales(np.array([a]), 1, col_scales=np.array([a]))[0, 0] == np.float32(1 + 2.0 ** -11)
    with pytest.raises(ValueError):
        O.element_scales(R, 7, group=3)  # 7 columns need 3 runs


def test_grouped_scales_hand_worked():
    # group 4 over 6 columns: runs [1, -2, 3, -4] and [8, 0.5]; no search: absmax / hi
    W = np.array([[1.0, -2.0, 3.0, -4.0, 8.0, 0.5]], dtype=np.float32)
    S, C = O.row_scales(W, -7, 7, 1, group=4)
    assert S.shape == (1, 2) and not C.any()
    assert S[0, 0] == np.float32(4.0 / 7.0) and S[0, 1] == np.float32(8.0 / 7.0)
    # a group of at least n columns is the per-row scale
    S1, _ = O.row_scales(W, -7, 7, 9, group=6)
    s, _ = O.row_scales(W, -7, 7, 9)
    assert S1.shape == (1, 1) and S1[0, 0] == s[0]


@pytest.mark.parametrize("m,n", [(3, 5), (5, 4), (7, 7)])
@pytest.mark.parametrize("bits", [0, 3, (-3, 3)])
def test_entry_scales_all_solvers_agree_with_naive(m, n, bits):
    """Theorem 3.2 with one scale per entry: the naive solve on vec(W) (its
    scales flattened column-major) and every ordered solver agree."""
    from workloads import random_problem

    p = random_problem(m, n, bits=0, seed=17 * m + n)
    rng = np.random.default_rng(m + 31 * n)
    R = rng.uniform(0.2, 0.6, (m, 2)).astype(np.float32)
    t = rng.uniform(0.5, 2.0, n).astype(np.float32)
    S = O.element_scales(R, n, group=(n + 1) // 2, col_scales=t)
    Vn, _, En = O.bakron_naive(p.W, p.A, p.B, S, bits)
    LA, LB = O.factors_of(p.A, p.B)
    for method in ENTRY_SOLVERS:
        V, Wq, E = _entry_solve(p.W, LA, LB, S, bits, method)
        assert np.array_equal(V, Vn), method
        assert np.allclose(E, En, atol=1e-11), method


@pytest.mark.parametrize("bits", [0, 2, (-3, 3)])
def test_entry_scales_with_diagonal_factors_round_each_entry(bits):
    """A, B diagonal: every entry is rounded on its own alphabet sigma_ij {lo..hi}."""
    from workloads import random_problem

    m, n = 6, 9
    p = random_problem(m, n, bits=0, seed=5, kind="diagonal")
    rng = np.random.default_rng(8)
    R = rng.uniform(0.1, 0.9, (m, 3)).astype(np.float32)
    t = rng.uniform(0.5, 2.0, n).astype(np.float32)
    S = O.element_scales(R, n, group=3, col_scales=t)
    rtn = np.rint((p.W.astype(np.float32) / S).astype(np.float32))
    b = O.alphabet_bounds(bits)
    if b is not None:
        rtn = np.clip(rtn, b[0], b[1])
    LA, LB = O.factors_of(p.A, p.B)
    for method in ENTRY_SOLVERS:
        V, Wq, _ = _entry_solve(p.W, LA, LB, S, bits, method)
        assert np.array_equal(V, rtn.astype(np.int64)), method
        assert np.array_equal(Wq, S.astype(np.float64) * V), method
    Vg, _, _ = O.gptq_rows(p.W, p.A, S, bits)
    assert np.array_equal(Vg, rtn.astype(np.int64))


@pytest.mark.parametrize("bits", [0, (-4, 3)])
def test_power_of_two_column_scales_are_a_change_of_variables(bits):
    """Column scales t_j = 2^k_j: the problem (W, A, B, s_i t_j) is the
    row-scaled problem (W D^-1, D A D, B, s_i) with D = diag(t) -- the
    objective tr((Wq - W) A (Wq - W)^T B) is the same after Wq = Wq' D --
    and every step of the solve scales exactly by powers of two, so the codes
    are identical."""
    from workloads import random_problem

    m, n = 6, 10
    p = random_problem(m, n, bits=0, seed=21)
    rng = np.random.default_rng(4)
    s = rng.uniform(0.2, 0.5, m).astype(np.float32)
    t = (2.0 ** rng.integers(-3, 4, n)).astype(np.float32)
    S = O.element_scales(s, n, col_scales=t)
    LA, LB = O.factors_of(p.A, p.B)
    V, Wq, _ = O.bakron(p.W, LA=LA, LB=LB, scales=S, bits=bits)
    D = np.diag(t.astype(np.float64))
    W2 = (p.W.astype(np.float64) / t[None, :]).astype(np.float32)
    LA2, LB2 = O.factors_of(D @ p.A.astype(np.float64) @ D, p.B)
    V2, Wq2, _ = O.bakron(W2, LA=LA2, LB=LB2, scales=s, bits=bits)
    assert np.array_equal(V, V2)
    assert np.array_equal(Wq, Wq2 * t[None, :])
    Vn, _, _ = O.bakron_naive(p.W, p.A, p.B, S, bits)
    assert np.array_equal(V, Vn)


def test_entry_scale_pins_catch_planted_mistakes(monkeypatch):
    """A scale read from the wrong column, or a row-major vec of the scale
    matrix, makes the per-entry rounding pin or the naive agreement fail."""
    import oracle.naive as N
    import oracle.recursive as R
    from workloads import random_problem

    m, n = 6, 9
    p = random_problem(m, n, bits=0, seed=5, kind="diagonal")
    rng = np.random.default_rng(8)
    S = O.element_scales(rng.uniform(0.1, 0.9, (m, 3)).astype(np.float32), n, group=3,
                         col_scales=rng.uniform(0.5, 2.0, n).astype(np.float32))
    expect = np.rint((p.W.astype(np.float32) / S).astype(np.float32)).astype(np.int64)
    LA, LB = O.factors_of(p.A, p.B)
    assert np.array_equal(O.bakron(p.W, LA=LA, LB=LB, scales=S, bits=0)[0], expect)

    def first_column_scale(scales, rows, cols):
        s = np.asarray(scales, dtype=np.float32)
        return s[rows] if s.ndim == 1 else s[rows, np.zeros_like(cols)]

    with monkeypatch.context() as mp:
        mp.setattr(R, "scale_at", first_column_scale)
        assert not np.array_equal(O.bakron(p.W, LA=LA, LB=LB, scales=S, bits=0)[0], expect)

    q = random_problem(5, 4, bits=0, seed=3)
    S2 = O.element_scales(rng.uniform(0.2, 0.6, (5, 2)).astype(np.float32), 4, group=2)
    Vn = O.bakron_naive(q.W, q.A, q.B, S2, 3)[0]
    assert np.array_equal(Vn, O.bakron(q.W, q.A, q.B, S2, 3)[0])
    with monkeypatch.context() as mp:
        mp.setattr(N, "_vec_scales", lambda s, m_, n_: np.asarray(s, np.float32).flatten(order="C"))
        assert not np.array_equal(O.bakron_naive(q.W, q.A, q.B, S2, 3)[0], Vn)
