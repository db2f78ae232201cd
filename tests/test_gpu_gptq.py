"""Row-wise GPTQ on the GPU (bakron_gptq_quantize, the one-sided case B = I
of the BaKron solve) against the oracle: Algorithm 1 with H = A on every row
("BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 1
and Sec. 3.1).  Same bar as the BaKron parity tests."""

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

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _gpu_gptq(bk, p):
    import torch

    LA, info = bk.factor(_dev(p.A))
    V, Wq, st = bk.gptq(_dev(p.W), LA, None if p.scales is None else _dev(p.scales), p.bits)
    torch.cuda.synchronize()
    assert int(info.item()) == 0 and int(st.item()) == 0
    return LA, V.cpu().numpy().astype(np.int64), Wq.cpu().numpy().astype(np.float64)


SHAPES = [(1, 1), (5, 3), (32, 32), (45, 70), (64, 64), (100, 37), (130, 257), (200, 96)]


@pytest.mark.parametrize("m,n", SHAPES)
@pytest.mark.parametrize("bits", [0, 2, 4])
def test_gptq_against_rowwise_oracle(bk, m, n, bits):
    p = random_problem(m, n, bits=bits, seed=m * 1000 + n + bits, kind="gram")
    _, V, Wq = _gpu_gptq(bk, p)
    Vo, Wqo, _ = O.gptq_rows(p.W, p.A, p.scales, p.bits)
    assert O.match_fraction(V, Vo) >= V_MATCH
    I = np.eye(m)
    d_ref = O.distortion(p.W, Wqo, p.A, I)
    d_gpu = O.distortion(p.W, Wq, p.A, I)
    assert abs(d_gpu - d_ref) <= distortion_tolerance(d_ref, Wqo, p.A, I, D_REL)


def test_gptq_equals_bakron_with_identity_output_factor(bk):
    import torch

    p = random_problem(150, 211, bits=3, seed=11, kind="gram")
    LA, V, Wq = _gpu_gptq(bk, p)
    eye = torch.eye(p.m, dtype=torch.float32, device="cuda")
    V2, Wq2, st = bk.quantize(_dev(p.W), LA, eye, _dev(p.scales), p.bits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(V, V2.cpu().numpy()) and np.array_equal(Wq, Wq2.cpu().numpy().astype(np.float64))


def test_gptq_c2_against_oracle(bk):
    p = make_config("c2")
    LA, V, Wq = _gpu_gptq(bk, p)
    LA64, _ = O.factors_of(p.A, np.eye(1, dtype=np.float32))
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=np.eye(p.m), scales=p.scales, bits=p.bits)
    assert O.match_fraction(V, Vo) >= V_MATCH
    I = np.eye(p.m)
    d_ref = O.distortion(p.W, Wqo, p.A, I)
    assert abs(O.distortion(p.W, Wq, p.A, I) - d_ref) <= D_REL * abs(d_ref)
