"""The seeded input generators: determinism, shapes and positive definiteness."""

import numpy as np
import pytest

from workloads import make_config, random_problem, row_absmax_scales


def test_c1_c2_deterministic_and_shaped():
    for key, (m, n, bits) in {"c1": (64, 64, 0), "c2": (1024, 1024, 4)}.items():
        p1, p2 = make_config(key), make_config(key)
        assert p1.digest() == p2.digest()
        assert (p1.m, p1.n, p1.bits) == (m, n, bits)
        assert p1.W.shape == (m, n) and p1.A.shape == (n, n) and p1.B.shape == (m, m)
        for M in (p1.A, p1.B):
            assert M.dtype == np.float32 and np.array_equal(M, M.T)
            assert np.linalg.eigvalsh(M.astype(np.float64)).min() > 0
        if bits:
            assert p1.scales.shape == (m,) and np.all(p1.scales > 0)
        else:
            assert p1.scales is None


def test_absmax_scale_rule():
    W = np.array([[0.7, -1.4, 0.0], [0.3, 0.1, -0.2]], dtype=np.float32)
    assert np.allclose(row_absmax_scales(W, 4), [1.4 / 7, 0.3 / 7])
    assert np.allclose(row_absmax_scales(W, 2), [1.4, 0.3])


@pytest.mark.parametrize("kind", ["gram", "identity_b", "diagonal", "ar1"])
def test_random_problem_kinds(kind):
    p = random_problem(7, 5, bits=3, seed=1, kind=kind)
    assert p.W.shape == (7, 5) and p.A.shape == (5, 5) and p.B.shape == (7, 7)
    assert np.linalg.eigvalsh(p.A.astype(np.float64)).min() > 0
    assert np.linalg.eigvalsh(p.B.astype(np.float64)).min() > 0


def test_bf16_encoding_rounds_to_nearest_even():
    from workloads.activations import from_bf16_bits, to_bf16_bits

    x = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -9, 1 + 2.0 ** -7 + 2.0 ** -8, -2.5, 0.0], np.float32)
    y = from_bf16_bits(to_bf16_bits(x))
    assert np.array_equal(y, np.array([1.0, 1.0, 1 + 2.0 ** -7, 1 + 2.0 ** -6, -2.5, 0.0], np.float32))


def test_samples_are_seeded_and_bf16_valued():
    from workloads.activations import from_bf16_bits, make_samples, to_bf16_bits

    s1, s2 = make_samples(6, 4, 9, seed=3), make_samples(6, 4, 9, seed=3)
    assert np.array_equal(s1.a_bits, s2.a_bits) and np.array_equal(s1.b_bits, s2.b_bits)
    assert np.array_equal(to_bf16_bits(s1.a_f32), s1.a_bits)
    assert s1.a_bits.shape == (6, 9) and s1.b_bits.shape == (4, 9)
