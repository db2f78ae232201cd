"""BaKron-antidiagonal on the GPU (bakron_antidiag_quantize; Algorithm 3 of
"BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 3.2)
against the oracle, at the BaKron parity bar: codes identical in at least
99.99% of the entries and the distortion within 1e-4 relative.  By
Theorem 3.2 its codes are BaKron's, so it is also compared with the GPU
BaKron solve."""

import numpy as np
import pytest

import oracle as O
from tolerances import distortion_tolerance
from workloads import make_config, random_problem

pytestmark = pytest.mark.gpu

V_MATCH = 0.9999
D_REL = 1e-4


@pytest.fixture(scope="module")
def bk():
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import build as b

    b.build()
    bk.load_library()
    torch.cuda.init()
    return bk


def _dev(x):
    import torch

    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _run(bk, p):
    import torch

    LA, LB, info = bk.prepare(_dev(p.A), _dev(p.B))
    assert info.cpu().tolist() == [0, 0]
    V, Wq, st = bk.antidiag(_dev(p.W), LA, LB, _dev(p.scales), p.bits)
    V2, _, st2 = bk.quantize(_dev(p.W), LA, LB, _dev(p.scales), p.bits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    return V.cpu().numpy().astype(np.int64), Wq.cpu().numpy(), V2.cpu().numpy().astype(np.int64)


def _check(p, V, Wq, Vb):
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=p.scales, bits=p.bits)
    assert O.match_fraction(V, Vo) >= V_MATCH
    assert O.match_fraction(V, Vb) >= V_MATCH
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    d_gpu = O.distortion(p.W, Wq.astype(np.float64), p.A, p.B)
    assert abs(d_gpu - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, p.B, D_REL)
    s = np.ones(p.m, np.float32) if p.scales is None else p.scales
    assert np.array_equal(Wq, (s[:, None] * V.astype(np.float32)).astype(np.float32))


SHAPES = [(1, 1), (1, 9), (9, 1), (3, 5), (31, 33), (32, 32), (33, 31), (65, 97), (100, 37), (130, 70)]


@pytest.mark.parametrize("m,n", SHAPES)
@pytest.mark.parametrize("bits", [0, 2, 4])
def test_antidiag_against_oracle(bk, m, n, bits):
    p = random_problem(m, n, bits=bits, seed=m * 1000 + n + bits)
    _check(p, *_run(bk, p))


@pytest.mark.parametrize("kind", ["ar1", "diagonal", "identity_b"])
def test_antidiag_special_factors(bk, kind):
    p = random_problem(48, 80, bits=3, seed=9, kind=kind)
    _check(p, *_run(bk, p))


def test_antidiag_ignores_the_upper_triangles(bk):
    """Entries above the diagonal of L_A, L_B are ignored and the diagonal is
    taken as 1 (the factors' documented contract)."""
    import torch

    p = random_problem(40, 50, bits=4, seed=4)
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    V1, Wq1, _ = bk.antidiag(_dev(p.W), LA, LB, _dev(p.scales), 4)
    LAg = LA + torch.triu(torch.full_like(LA, 7.0))
    LBg = LB + torch.triu(torch.full_like(LB, -5.0))
    V2, Wq2, st = bk.antidiag(_dev(p.W), LAg, LBg, _dev(p.scales), 4)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(V1, V2) and torch.equal(Wq1, Wq2)


def test_antidiag_flags_nonfinite_weights(bk):
    import torch

    p = random_problem(20, 30, bits=4, seed=1)
    W = p.W.copy()
    W[3, 4] = np.nan
    LA, LB, _ = bk.prepare(_dev(p.A), _dev(p.B))
    _, _, st = bk.antidiag(_dev(W), LA, LB, _dev(p.scales), 4)
    torch.cuda.synchronize()
    assert int(st.item()) & 1  # BAKRON_DEV_NONFINITE_W


def test_antidiag_c2_against_oracle(bk):
    """The 1024 x 1024 int4 workload in full."""
    p = make_config("c2")
    _check(p, *_run(bk, p))


def test_antidiag_c3_equals_bakron(bk):
    """The 4096 x 4096 int4 workload (about 20 s of Algorithm 3): by
    Theorem 3.2 the codes equal the BaKron solve's, whose own full-size
    parity with the oracle is tested separately; here every code is compared
    with BaKron's and the first 8 rows with the oracle's (a row's codes do
    not depend on later rows, so the oracle solves those rows alone, with the
    leading block of L_B)."""
    p = make_config("c3")
    V, Wq, Vb = _run(bk, p)
    assert O.match_fraction(V, Vb) >= V_MATCH
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, _, _ = O.bakron(p.W[:8], LA=LA64, LB=LB64[:8, :8], scales=None if p.scales is None else p.scales[:8],
                        bits=p.bits)
    assert O.match_fraction(V[:8], Vo) >= V_MATCH
