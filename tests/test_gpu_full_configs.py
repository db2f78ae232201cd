"""Full-size workloads through the C ABI, in the configuration the benchmark
times (bakron_prepare + bakron_quantize on the device), against the fp64
oracle entry by entry: c3 (4096 x 4096), c4 (14336 x 4096), c5 (4096 x 14336);
the persistent solve (bakron_quantize_persistent) on the same factors is
held to the same bars against the same oracle codes.

For each workload the GPU factors L-hat_A, L-hat_B are compared with the
oracle's (Cholesky of the inverse in fp64, "BaKron: Efficient Quantization
with Kronecker-Factored Hessians", Sec. 3.2, Algorithm 1) within the bound
that the double-float unit and cond(H) give (tests/tolerances.py), and the
codes with the oracle's Alg. 5 solve from those fp64 factors (App. B eq. (2)
defines the one correct V): at least 99.99% identical, distortion within
1e-4 relative.  Each case takes one to two minutes of host time (input
generation and the oracle on the host cores).

Ragged shapes that reach the chunk products of the solve (more than two
chunks of tile rows and columns, edges not multiples of 32) are compared the
same way: below 2^22 weights (digits made in the chunk kernel), between 2^22
and 2^24 (packed factor digits, items shared evenly over the CTAs), and
above 2^24 (packed digits, one candidate per CTA).
"""

import numpy as np
import pytest

import oracle as O
from tolerances import check_factor, distortion_tolerance
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


def _solve(bk, p):
    """GPU factors, then the solve by bakron_quantize and by
    bakron_quantize_persistent on those factors."""
    import torch

    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()  # noqa: E731
    LA, LB, info = bk.prepare(dev(p.A), dev(p.B))
    W, s = dev(p.W), None if p.scales is None else dev(p.scales)
    out = {}
    for name, solve in (("wavefront", bk.quantize), ("persistent", bk.quantize_persistent)):
        V, Wq, st = solve(W, LA, LB, s, p.bits)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, name
        out[name] = (V.cpu().numpy().astype(np.int64), Wq.cpu().numpy())
    assert info.cpu().tolist() == [0, 0]
    return LA.cpu().numpy(), LB.cpu().numpy(), out


def _against_oracle(bk, p):
    """Asserts the bars and prints one line per solve (pytest -s shows them):
    codes identical, distortions, and the factors' largest error as a
    fraction of their bound."""
    LA, LB, out = _solve(bk, p)
    LA64, LB64 = O.factors_of(p.A, p.B)
    fa = check_factor(LA, LA64, p.A)
    fb = check_factor(LB, LB64, p.B)
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=p.scales, bits=p.bits)
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    tol = distortion_tolerance(d_ref, Wqo, p.A, p.B, D_REL)
    for name, (V, Wq) in out.items():
        match = O.match_fraction(V, Vo)
        d_gpu = O.distortion(p.W, Wq.astype(np.float64), p.A, p.B)
        same = int(np.count_nonzero(V == Vo))
        print(f"\nparity {p.name} {p.m}x{p.n} b{p.bits} {name}: codes identical {same} of {V.size} ({match:.8f}); "
              f"distortion {d_gpu:.10g} vs oracle {d_ref:.10g} (rel {abs(d_gpu - d_ref) / max(abs(d_ref), 1e-300):.2g}); "
              f"factor error / bound: L_A {fa:.3g}, L_B {fb:.3g}")
        assert match >= V_MATCH, (p.name, name, match)
        assert abs(d_gpu - d_ref) <= tol, (p.name, name, d_gpu, d_ref)


@pytest.mark.parametrize("key", ["c2", "c3", "c4", "c5"])
def test_full_size_against_oracle(bk, key):
    _against_oracle(bk, make_config(key))


@pytest.mark.parametrize("m,n,bits", [(1000, 1300, 3), (1300, 1000, 3), (2100, 2100, 4), (4100, 4100, 4)])
def test_ragged_chunk_shapes_against_oracle(bk, m, n, bits):
    # 2100 x 2100 = 4.41 M weights >= 2^22: packed digits, shared items;
    # 4100 x 4100 = 16.81 M weights > 2^24: packed digits, one candidate per CTA.
    _against_oracle(bk, random_problem(m, n, bits=bits, seed=m + 7 * n, w_std=0.02))
