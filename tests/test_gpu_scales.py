"""The base quantizer's variants on the GPU against the oracle ("BaKron:
Efficient Quantization with Kronecker-Factored Hessians", App. D: per-row
scales with an MSE shrink search; Sec. 3.1: integer alphabets):

* bakron_row_scales against oracle.row_scales: grid 1 bit-identical; with a
  search, the same shrink factor on at least 99.9% of the rows, and where the
  choice differs the two candidates' errors (the oracle's fp64 sums) within
  1e-9 relative -- a tie the two summation orders may break differently;
* bakron_pack_codes against oracle.pack_codes: byte-identical;
* bakron_quantize_range (explicit alphabets {lo .. hi}, with and without
  L_B) against the oracle's solve over the same alphabet, at the BaKron
  parity bar; bits = b is the alphabet {-2^(b-1) .. 2^(b-1) - 1}
  bit-identically.
"""

import numpy as np
import pytest

import oracle as O
from tolerances import distortion_tolerance
from workloads import make_config, random_problem

pytestmark = pytest.mark.gpu

V_MATCH = 0.9999
D_REL = 1e-4
G_MATCH = 0.999
ERR_TIE = 1e-9


@pytest.fixture(scope="module")
def bk():
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import build as b

    b.build()
    bk.load_library()
    torch.cuda.init()
    return bk


def _dev(x, dtype=None):
    import torch

    if x is None:
        return None
    a = np.ascontiguousarray(x, dtype=np.float32 if dtype is None else dtype)
    return torch.from_numpy(a).cuda()


def _check_scales(W, lo, hi, grid, Sg):
    """Sg (the GPU's scales) against the oracle on every row of W."""
    So, chosen = O.row_scales(W, lo, hi, grid)
    if grid == 1:
        assert np.array_equal(Sg, So)
        return
    f = O.shrink_factors(grid)
    same = Sg == So
    assert same.mean() >= G_MATCH, same.mean()
    for i in np.flatnonzero(~same):
        # the GPU's scale is one of the row's candidates, tied with the oracle's choice
        s0 = np.float32(np.float32(np.max(np.abs(W[i]))) / np.float32(hi))
        assert Sg[i] in (s0 * f).astype(np.float32), (i, Sg[i], s0)
        e_o = O.row_error(W[i], So[i], lo, hi)
        e_g = O.row_error(W[i], Sg[i], lo, hi)
        assert e_g <= e_o * (1 + ERR_TIE), (i, chosen[i], e_g, e_o)


@pytest.mark.parametrize("m,n", [(1, 1), (7, 3), (64, 257), (300, 1000), (33, 4099)])
@pytest.mark.parametrize("alphabet", [(-8, 7), (-7, 7), (-2, 1)])
@pytest.mark.parametrize("grid", [1, 2, 20, 100])
def test_row_scales_against_oracle(bk, m, n, alphabet, grid):
    import torch

    rng = np.random.default_rng(m * 7919 + n * 31 + grid + alphabet[0] * 3 + alphabet[1])
    W = rng.standard_normal((m, n)).astype(np.float32)
    # heavy-tailed rows: an outlier per row makes the shrink search matter
    W[:, 0] *= 8.0
    lo, hi = alphabet
    Sg = bk.row_scales(_dev(W), lo, hi, grid)
    torch.cuda.synchronize()
    _check_scales(W, lo, hi, grid, Sg.cpu().numpy())


def test_row_scales_special_rows(bk):
    import torch

    n = 40
    W = np.zeros((6, n), dtype=np.float32)
    W[1] = 0.375  # constant row
    W[2, 17] = -3.0  # a single nonzero
    W[3] = np.linspace(-1, 1, n, dtype=np.float32)
    W[4, ::2] = 1e-30  # tiny magnitudes (normal floats near the bottom of the range)
    W[5] = np.float32(2.0) ** np.arange(-20, 20, dtype=np.float32)  # wide dynamic range
    for lo, hi in [(-8, 7), (-1, 1)]:
        for grid in (1, 3, 50):
            Sg = bk.row_scales(_dev(W), lo, hi, grid)
            torch.cuda.synchronize()
            Sg = Sg.cpu().numpy()
            assert Sg[0] == 1.0
            _check_scales(W, lo, hi, grid, Sg)


def test_row_scales_long_rows_read_from_global_memory(bk):
    """Rows longer than the shared-memory staging limit take the L2 path."""
    import torch

    rng = np.random.default_rng(5)
    W = rng.standard_normal((3, 60001)).astype(np.float32)
    Sg = bk.row_scales(_dev(W), -8, 7, 12)
    torch.cuda.synchronize()
    _check_scales(W, -8, 7, 12, Sg.cpu().numpy())


def test_row_scales_full_size_sampled_rows(bk):
    """The 4096 x 4096 workload's weights, grid 100: every GPU scale is
    checked against the oracle on a sample of 64 rows."""
    import torch

    p = make_config("c3")
    Sg = bk.row_scales(_dev(p.W), -8, 7, 100)
    torch.cuda.synchronize()
    Sg = Sg.cpu().numpy()
    rows = np.random.default_rng(3).choice(p.m, 64, replace=False)
    _check_scales(p.W[rows], -8, 7, 100, Sg[rows])


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("m,n", [(1, 1), (3, 5), (17, 33), (64, 1001), (257, 64)])
def test_pack_codes_against_oracle(bk, bits, m, n):
    import torch

    rng = np.random.default_rng(bits * 100 + m + n)
    half = 1 << (bits - 1)
    V = rng.integers(-half, half, size=(m, n)).astype(np.int32)
    Pg = bk.pack_codes(_dev(V, np.int32), bits)
    torch.cuda.synchronize()
    Pg = Pg.cpu().numpy()
    Po = O.pack_codes(V, bits)
    assert Pg.dtype == np.uint8 and Pg.shape == Po.shape
    assert np.array_equal(Pg, Po)
    assert np.array_equal(O.unpack_codes(Pg, n, bits), V)


def _range_gpu(bk, p, LB, lo, hi, scales):
    import torch

    LA, LBg, info = bk.prepare(_dev(p.A), _dev(p.B))
    assert info.cpu().tolist() == [0, 0]
    V, Wq, st = bk.quantize_range(_dev(p.W), LA, LBg if LB else None, _dev(scales), lo, hi)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return V.cpu().numpy().astype(np.int64), Wq.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("m,n", [(5, 3), (45, 70), (130, 257)])
@pytest.mark.parametrize("alphabet", [(-7, 7), (-1, 1), (0, 15), (-1000, 1000)])
def test_quantize_range_against_oracle(bk, m, n, alphabet):
    lo, hi = alphabet
    p = random_problem(m, n, bits=0, seed=m * 31 + n + hi)
    S, _ = O.row_scales(p.W, -hi if lo == 0 else lo, hi, 10)
    V, Wq = _range_gpu(bk, p, True, lo, hi, S)
    assert V.min() >= lo and V.max() <= hi
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=S, bits=(lo, hi))
    assert O.match_fraction(V, Vo) >= V_MATCH
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    d_gpu = O.distortion(p.W, Wq, p.A, p.B)
    assert abs(d_gpu - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, p.B, D_REL)
    assert np.array_equal(Wq.astype(np.float32), (S[:, None] * V.astype(np.float32)).astype(np.float32))


@pytest.mark.parametrize("alphabet", [(-7, 7), (-3, 4)])
def test_quantize_range_rowwise_against_oracle(bk, alphabet):
    """LB = NULL: the row-wise GPTQ solve over an explicit alphabet."""
    lo, hi = alphabet
    p = random_problem(96, 150, bits=0, seed=hi * 5 - lo)
    S, _ = O.row_scales(p.W, lo, hi, 1)
    V, Wq = _range_gpu(bk, p, False, lo, hi, S)
    Vo, Wqo, _ = O.gptq_rows(p.W, p.A, S, (lo, hi))
    assert O.match_fraction(V, Vo) >= V_MATCH
    I = np.eye(p.m)
    d_ref = O.distortion(p.W, Wqo, p.A, I)
    d_gpu = O.distortion(p.W, Wq, p.A, I)
    assert abs(d_gpu - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, I, D_REL)


def test_quantize_range_equals_bits_alphabet(bk):
    import torch

    p = random_problem(70, 90, bits=4, seed=23)
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    V1, Wq1, s1 = bk.quantize(_dev(p.W), LA, LB, _dev(p.scales), 4)
    V2, Wq2, s2 = bk.quantize_range(_dev(p.W), LA, LB, _dev(p.scales), -8, 7)
    torch.cuda.synchronize()
    assert int(s1.item()) == 0 and int(s2.item()) == 0
    assert torch.equal(V1, V2) and torch.equal(Wq1, Wq2)


def test_scales_solve_pack_end_to_end(bk):
    """The base quantizer of App. D end to end on the GPU: searched scales,
    the BaKron solve over {-8 .. 7}, the codes packed to 4 bits; checked
    against the oracle's codes and packing."""
    import torch

    p = random_problem(64, 128, bits=0, seed=99)
    W = _dev(p.W)
    S = bk.row_scales(W, -8, 7, 20)
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    V, Wq, st = bk.quantize_range(W, LA, LB, S, -8, 7)
    P = bk.pack_codes(V, 4)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Sg = S.cpu().numpy()
    _check_scales(p.W, -8, 7, 20, Sg)
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, _, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=Sg, bits=(-8, 7))
    Vg = V.cpu().numpy()
    assert O.match_fraction(Vg, Vo) >= V_MATCH
    assert np.array_equal(P.cpu().numpy(), O.pack_codes(Vg, 4))


@pytest.mark.parametrize("m,n,group", [(5, 9, 4), (64, 1000, 128), (20, 300, 300), (3, 70000, 60001)])
def test_grouped_scales_against_oracle(bk, m, n, group):
    """One scale per run of `group` columns; each run checked like a row."""
    import torch

    rng = np.random.default_rng(m + n + group)
    W = rng.standard_normal((m, n)).astype(np.float32)
    W[:, ::97] *= 6.0
    Sg = bk.row_scales(_dev(W), -4, 3, 16, group=group)
    torch.cuda.synchronize()
    Sg = Sg.cpu().numpy()
    runs = -(-n // group)
    assert Sg.shape == (m, runs)
    for k in range(runs):
        _check_scales(W[:, k * group:(k + 1) * group], -4, 3, 16, Sg[:, k])


def _scaled_case(m, n, group, with_cols, seed):
    p = random_problem(m, n, bits=0, seed=seed)
    rng = np.random.default_rng(seed + 1)
    R = None
    if group is not None or not with_cols:
        R, _ = O.row_scales(p.W, -7, 7, 8, group=group)
    t = rng.uniform(0.5, 2.0, n).astype(np.float32) if with_cols else None
    S = O.element_scales(np.ones(m, np.float32) if R is None else R, n, group=group, col_scales=t)
    return p, R, t, S


@pytest.mark.parametrize("m,n", [(5, 3), (45, 70), (130, 257)])
@pytest.mark.parametrize("group,with_cols", [(32, False), (16, True), (None, True), (100, True)])
@pytest.mark.parametrize("with_lb", [True, False])
def test_quantize_scaled_against_oracle(bk, m, n, group, with_cols, with_lb):
    import torch

    p, R, t, S = _scaled_case(m, n, group, with_cols, seed=m * 13 + n + (group or 0))
    LA, LB, info = bk.prepare(_dev(p.A), _dev(p.B))
    assert info.cpu().tolist() == [0, 0]
    V, Wq, st = bk.quantize_scaled(_dev(p.W), LA, LB if with_lb else None, _dev(R), -7, 7, group=group,
                                   col_scales=_dev(t))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    V = V.cpu().numpy().astype(np.int64)
    Wq = Wq.cpu().numpy()
    assert np.array_equal(Wq, (S * V.astype(np.float32)).astype(np.float32))
    if with_lb:
        LA64, LB64 = O.factors_of(p.A, p.B)
        Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=S, bits=(-7, 7))
        Bm = p.B
    else:
        Vo, Wqo, _ = O.gptq_rows(p.W, p.A, S, (-7, 7))
        Bm = np.eye(m)
    assert O.match_fraction(V, Vo) >= V_MATCH
    d_ref = O.distortion(p.W, Wqo, p.A, Bm)
    d_gpu = O.distortion(p.W, Wq.astype(np.float64), p.A, Bm)
    assert abs(d_gpu - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, Bm, D_REL)


def test_quantize_scaled_defaults_equal_range(bk):
    """No groups and no column scales is bakron_quantize_range bit for bit."""
    import torch

    p = random_problem(70, 90, bits=4, seed=29)
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    V1, Wq1, s1 = bk.quantize_range(_dev(p.W), LA, LB, _dev(p.scales), -8, 7)
    V2, Wq2, s2 = bk.quantize_scaled(_dev(p.W), LA, LB, _dev(p.scales), -8, 7)
    torch.cuda.synchronize()
    assert int(s1.item()) == 0 and int(s2.item()) == 0
    assert torch.equal(V1, V2) and torch.equal(Wq1, Wq2)


def test_quantize_scaled_rejects_bad_column_scales(bk):
    import torch

    p = random_problem(20, 30, bits=4, seed=2)
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    t = np.ones(30, np.float32)
    t[7] = 0.0
    _, _, st = bk.quantize_scaled(_dev(p.W), LA, LB, _dev(p.scales), -8, 7, col_scales=_dev(t))
    torch.cuda.synchronize()
    assert int(st.item()) & 2  # BAKRON_DEV_BAD_SCALE


def test_quantize_scaled_multi_tile_grouped(bk):
    """Groups of 128 and column scales over many tiles and chunks (520 x 700,
    ragged in both dimensions), BaKron with both factors."""
    import torch

    p, R, t, S = _scaled_case(520, 700, 128, True, seed=77)
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    V, Wq, st = bk.quantize_scaled(_dev(p.W), LA, LB, _dev(R), -7, 7, group=128, col_scales=_dev(t))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=S, bits=(-7, 7))
    V = V.cpu().numpy().astype(np.int64)
    assert O.match_fraction(V, Vo) >= V_MATCH
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    d_gpu = O.distortion(p.W, Wq.cpu().numpy().astype(np.float64), p.A, p.B)
    assert abs(d_gpu - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, p.B, D_REL)
