"""GPU parity of the persistent solve, bakron_quantize_persistent (through
the C ABI), against the fp64 oracle: the same codes that App. B eq. (2)
defines ("BaKron: Efficient Quantization with Kronecker-Factored Hessians";
Theorem 3.2: every order of the anti-diagonals that respects the
dependencies gives that V), at the same bars as bakron_quantize: V identical
in at least 99.99% of the entries, distortion within 1e-4 relative plus the
effect of the final fp32 rounding of s*v.  The full-size workloads run in
tests/test_gpu_full_configs.py beside bakron_quantize.
"""

import numpy as np
import pytest

import oracle as O
from test_gpu_parity import SHAPES, _dev, check_against_oracle, gpu_prepare
from workloads import make_config, random_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bk():
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import build as b

    b.build()
    bk.load_library()
    torch.cuda.init()
    return bk


def persistent(bk, p, LA, LB):
    import torch

    V, Wq, status = bk.quantize_persistent(_dev(p.W), LA, LB, _dev(p.scales), p.bits)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return V.cpu().numpy().astype(np.int64), Wq.cpu().numpy()


@pytest.mark.parametrize("m,n", SHAPES + [(200, 300), (300, 200), (257, 129)])
@pytest.mark.parametrize("bits", [0, 3, 4])
def test_persistent_with_oracle_factors(bk, m, n, bits):
    p = random_problem(m, n, bits=bits, seed=7 * m + n + bits)
    LA64, LB64 = O.factors_of(p.A, p.B)
    LA32, LB32 = LA64.astype(np.float32), LB64.astype(np.float32)
    Vg, Wqg = persistent(bk, p, _dev(LA32), _dev(LB32))
    check_against_oracle(p, Vg, Wqg, LA32.astype(np.float64), LB32.astype(np.float64), f"{m}x{n} b{bits}")


@pytest.mark.parametrize("m,n,bits,kind", [(40, 50, 3, "identity_b"), (50, 40, 4, "diagonal"), (70, 33, 0, "ar1"),
                                           (96, 96, 8, "gram")])
def test_persistent_special_cases(bk, m, n, bits, kind):
    p = random_problem(m, n, bits=bits, seed=11, kind=kind)
    LA, LB = gpu_prepare(bk, p)
    Vg, Wqg = persistent(bk, p, LA, LB)
    check_against_oracle(p, Vg, Wqg, *O.factors_of(p.A, p.B), f"{kind} {m}x{n}")


@pytest.mark.parametrize("key", ["c1", "c2"])
def test_persistent_workloads(bk, key):
    p = make_config(key)
    LA, LB = gpu_prepare(bk, p)
    Vg, Wqg = persistent(bk, p, LA, LB)
    check_against_oracle(p, Vg, Wqg, *O.factors_of(p.A, p.B), key)


def test_persistent_status_word_flags_bad_inputs(bk):
    import torch

    p = random_problem(20, 30, bits=4, seed=1)
    LA64, LB64 = O.factors_of(p.A, p.B)
    LA, LB = _dev(LA64), _dev(LB64)
    W = p.W.copy()
    W[3, 4] = np.inf
    _, _, st = bk.quantize_persistent(_dev(W), LA, LB, _dev(p.scales), 4)
    torch.cuda.synchronize()
    assert int(st.item()) & 1
