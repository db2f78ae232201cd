"""Full-size workloads c3, c4, c5 through the C ABI, in the configuration the
benchmark times (bakron_prepare + bakron_quantize on the device).

c3 (4096 x 4096) is compared with the fp64 oracle entry by entry.  c4 and c5
(14336 x 4096, 4096 x 14336) are checked by a property that holds at any
size and pins the result: given the GPU's codes, the errors they imply are
E = L_B^-1 (Wq - W) L_A^-T (App. B eq. (1)), the values the entries were
rounded at are W~ = Wq - E, and every code must be the alphabet's nearest
value to its W~ (the defining rule of App. B eq. (2)).  A V that passes this
for every entry is the unique BaKron output; entries whose W~/s lies within
1e-6 of a rounding tie are exempt.  With BAKRON_FULL_PARITY=1 in the
environment, c4 and c5 are compared with the fp64 oracle as well (minutes of
host time each).
"""

import os

import numpy as np
import pytest

import oracle as O
from workloads import make_config

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
    import torch

    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()  # noqa: E731
    LA, LB, info = bk.prepare(dev(p.A), dev(p.B))
    V, Wq, st = bk.quantize(dev(p.W), LA, LB, None if p.scales is None else dev(p.scales), p.bits)
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0, 0] and int(st.item()) == 0
    return LA.cpu().numpy(), LB.cpu().numpy(), V.cpu().numpy().astype(np.int64), Wq.cpu().numpy()


def nearest_rule_violations(p, V, LA64, LB64):
    """(fraction of codes that are not the nearest alphabet value, count of
    near-ties exempted, the implied errors E)."""
    s = np.ones(p.m, np.float32) if p.scales is None else p.scales
    Wq = s.astype(np.float64)[:, None] * V  # exact s * v, as the solve forms it
    E = O.errors_from_output(p.W, Wq, LA64, LB64)
    Wt = Wq - E
    y = (Wt.astype(np.float32) / s[:, None]).astype(np.float32)
    v = np.rint(y)
    if p.bits:
        v = np.clip(v, -(1 << (p.bits - 1)), (1 << (p.bits - 1)) - 1)
    tie = np.abs(y - np.floor(y) - 0.5) < 1e-6
    bad = (v.astype(np.int64) != V) & ~tie
    return float(bad.mean()), int(tie.sum()), E


def test_c3_against_oracle(bk):
    p = make_config("c3")
    LA, LB, V, Wq = _solve(bk, p)
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=p.scales, bits=p.bits)
    assert O.match_fraction(V, Vo) >= V_MATCH
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    assert abs(O.distortion(p.W, Wq.astype(np.float64), p.A, p.B) - d_ref) <= D_REL * abs(d_ref)


@pytest.mark.parametrize("key", ["c4", "c5"])
def test_full_size_nearest_rule(bk, key):
    p = make_config(key)
    LA, LB, V, Wq = _solve(bk, p)
    frac, ties, E = nearest_rule_violations(p, V, LA.astype(np.float64), LB.astype(np.float64))
    assert frac <= 1.0 - V_MATCH, (key, frac)
    assert ties <= 1e-5 * V.size, (key, ties)
    # the two exact forms of the distortion agree for the GPU's own errors
    s = np.ones(p.m) if p.scales is None else p.scales.astype(np.float64)
    d1 = O.distortion(p.W, s[:, None] * V, p.A, p.B)
    assert abs(d1 - O.distortion_from_errors(E, p.A, p.B)) <= 1e-6 * d1


@pytest.mark.skipif(os.environ.get("BAKRON_FULL_PARITY") != "1", reason="set BAKRON_FULL_PARITY=1 (minutes per case)")
@pytest.mark.parametrize("key", ["c4", "c5"])
def test_full_size_against_oracle(bk, key):
    p = make_config(key)
    LA, LB, V, Wq = _solve(bk, p)
    LA64, LB64 = O.factors_of(p.A, p.B)
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=p.scales, bits=p.bits)
    assert O.match_fraction(V, Vo) >= V_MATCH
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    assert abs(O.distortion(p.W, Wq.astype(np.float64), p.A, p.B) - d_ref) <= D_REL * abs(d_ref)
