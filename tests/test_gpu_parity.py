"""GPU parity: libbakron (through the C ABI) against the fp64 oracle.

Bars (the solver's stated tolerance): integer codes V identical in at least
99.99% of the entries, and the distortion tr(A (Wq-W)^T B (Wq-W)) within
1e-4 relative of the oracle's plus the effect of the final fp32 rounding of
s*v; the factors L-hat within the bound that the double-float unit and
cond(H) give (both bounds derived in tests/tolerances.py).
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


def _dev(x):
    import torch

    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def gpu_prepare(bk, p):
    LA, LB, info = bk.prepare(_dev(p.A), _dev(p.B))
    assert info.cpu().tolist() == [0, 0]
    return LA, LB


def gpu_quantize(bk, p, LA, LB):
    import torch

    V, Wq, status = bk.quantize(_dev(p.W), LA, LB, _dev(p.scales), p.bits)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return V.cpu().numpy().astype(np.int64), Wq.cpu().numpy()


def check_against_oracle(p, Vg, Wqg, LA64, LB64, label):
    Vo, Wqo, _ = O.bakron(p.W, LA=LA64, LB=LB64, scales=p.scales, bits=p.bits)
    match = O.match_fraction(Vg, Vo)
    d_ref = O.distortion(p.W, Wqo, p.A, p.B)
    d_gpu = O.distortion(p.W, Wqg.astype(np.float64), p.A, p.B)
    assert match >= V_MATCH, f"{label}: V match {match}"
    tol = distortion_tolerance(d_ref, Wqo, p.A, p.B, D_REL)
    assert abs(d_gpu - d_ref) <= tol, f"{label}: distortion {d_gpu} vs {d_ref}"
    s = np.ones(p.m, np.float32) if p.scales is None else p.scales
    assert np.array_equal(Wqg, (s[:, None] * Vg.astype(np.float32)).astype(np.float32))
    return match


SHAPES = [(1, 1), (1, 9), (9, 1), (3, 5), (17, 33), (31, 33), (32, 32), (33, 31), (64, 64), (65, 97), (100, 37),
          (130, 70)]


@pytest.mark.parametrize("m,n", SHAPES)
def test_factor_matches_oracle(bk, m, n):
    p = random_problem(m, n, bits=4, seed=m * 1000 + n)
    LA, LB = gpu_prepare(bk, p)
    LA64, LB64 = O.factors_of(p.A, p.B)
    check_factor(LA.cpu().numpy(), LA64, p.A)
    check_factor(LB.cpu().numpy(), LB64, p.B)


@pytest.mark.parametrize("m,n", SHAPES)
@pytest.mark.parametrize("bits", [0, 2, 4])
def test_quantize_with_oracle_factors(bk, m, n, bits):
    """Quantize alone: the GPU gets the oracle's factors rounded to fp32 and
    the oracle runs on the very same (promoted) factors."""
    p = random_problem(m, n, bits=bits, seed=7 * m + n + bits)
    LA64, LB64 = O.factors_of(p.A, p.B)
    LA32, LB32 = LA64.astype(np.float32), LB64.astype(np.float32)
    Vg, Wqg = gpu_quantize(bk, p, _dev(LA32), _dev(LB32))
    check_against_oracle(p, Vg, Wqg, LA32.astype(np.float64), LB32.astype(np.float64), f"{m}x{n} b{bits}")


@pytest.mark.parametrize("m,n,bits,kind", [(40, 50, 3, "identity_b"), (50, 40, 4, "diagonal"), (70, 33, 0, "ar1"),
                                           (96, 96, 8, "gram"), (33, 65, 3, "gram")])
def test_end_to_end_special_cases(bk, m, n, bits, kind):
    p = random_problem(m, n, bits=bits, seed=11, kind=kind)
    LA, LB = gpu_prepare(bk, p)
    Vg, Wqg = gpu_quantize(bk, p, LA, LB)
    LA64, LB64 = O.factors_of(p.A, p.B)
    check_against_oracle(p, Vg, Wqg, LA64, LB64, f"{kind} {m}x{n}")
    if kind == "diagonal":
        y = (p.W / p.scales[:, None]).astype(np.float32)
        rtn = np.clip(np.rint(y), -(1 << (bits - 1)), (1 << (bits - 1)) - 1)
        assert np.array_equal(Vg, rtn.astype(np.int64))


@pytest.mark.parametrize("key", ["c1", "c2"])
def test_workload_end_to_end(bk, key):
    """Workloads c1 (64 x 64, Z) and c2 (1024 x 1024, 4-bit): GPU prepare +
    quantize against the oracle from A, B."""
    p = make_config(key)
    LA, LB = gpu_prepare(bk, p)
    LA64, LB64 = O.factors_of(p.A, p.B)
    check_factor(LA.cpu().numpy(), LA64, p.A)
    check_factor(LB.cpu().numpy(), LB64, p.B)
    Vg, Wqg = gpu_quantize(bk, p, LA, LB)
    check_against_oracle(p, Vg, Wqg, LA64, LB64, key)


def test_status_word_flags_bad_inputs(bk):
    import torch

    p = random_problem(20, 30, bits=4, seed=1)
    LA64, LB64 = O.factors_of(p.A, p.B)
    LA, LB = _dev(LA64), _dev(LB64)
    W = p.W.copy()
    W[3, 4] = np.nan
    _, _, st = bk.quantize(_dev(W), LA, LB, _dev(p.scales), 4)
    torch.cuda.synchronize()
    assert int(st.item()) & 1
    s = p.scales.copy()
    s[5] = 0.0
    _, _, st = bk.quantize(_dev(p.W), LA, LB, _dev(s), 4)
    torch.cuda.synchronize()
    assert int(st.item()) & 2
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        bk.quantize(_dev(p.W), LA, LB, _dev(p.scales), 1)


def test_factor_reports_non_positive_pivot(bk):
    import torch

    H = np.eye(40, dtype=np.float32)
    H[7, 7] = -1.0  # the factorization runs from the last index backwards
    L, info = bk.factor(_dev(H))
    torch.cuda.synchronize()
    assert int(info.item()) == 1 + 7


def test_host_entry_point_matches_device_entry_point(bk):
    import torch

    p = random_problem(77, 45, bits=3, seed=5)
    LA64, LB64 = O.factors_of(p.A, p.B)
    LA32, LB32 = LA64.astype(np.float32), LB64.astype(np.float32)
    Vd, Wqd = gpu_quantize(bk, p, _dev(LA32), _dev(LB32))
    Vh, Wqh, st = bk.quantize_host(torch.from_numpy(p.W), torch.from_numpy(LA32), torch.from_numpy(LB32),
                                   torch.from_numpy(p.scales), p.bits)
    assert st == 0
    assert np.array_equal(Vh.numpy(), Vd) and np.array_equal(Wqh.numpy(), Wqd)


def test_bounded_wait_reports_a_timeout_and_the_context_survives(bk):
    """The tensor-core kernels' bounded mbarrier wait, run on a barrier that
    nothing arrives on: the device status reads BAKRON_DEV_TIMEOUT, and a
    solve afterwards still runs and matches the oracle."""
    import torch

    from kronecker_hessian_gptq_gb300 import _lib

    lib = bk.load_library()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.check(lib.bakron_selftest_wait_timeout(status.data_ptr(), torch.cuda.current_stream().cuda_stream),
               "bakron_selftest_wait_timeout")
    torch.cuda.synchronize()
    assert int(status.item()) == 4  # BAKRON_DEV_TIMEOUT
    p = random_problem(40, 50, bits=4, seed=8)
    LA, LB = gpu_prepare(bk, p)
    V, Wq = gpu_quantize(bk, p, LA, LB)
    check_against_oracle(p, V, Wq, *O.factors_of(p.A, p.B), "after timeout")


def test_profile_runs_the_tile_wavefront(bk):
    """bakron_quantize (and its profiled twin) runs the launch-per-step tile
    wavefront: tile solves, mid pushes and chunk products (classes 1..3),
    never the persistent sweep (class 4, bakron_quantize_persistent)."""
    import ctypes

    import torch

    from kronecker_hessian_gptq_gb300 import _lib

    lib = bk.load_library()
    p = random_problem(400, 300, bits=4, seed=12)
    LA64, LB64 = O.factors_of(p.A, p.B)
    W, LA, LB, s = _dev(p.W), _dev(LA64), _dev(LB64), _dev(p.scales)
    ws = torch.empty(bk.quantize_workspace_size(p.m, p.n), dtype=torch.uint8, device="cuda")
    V = torch.empty((p.m, p.n), dtype=torch.int32, device="cuda")
    Wq = torch.empty((p.m, p.n), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nc = len(_lib.KERNEL_CLASSES)
    kms, kl, kf = (ctypes.c_double * nc)(), (ctypes.c_int64 * nc)(), (ctypes.c_double * nc)()
    rc = lib.bakron_quantize_profile(W.data_ptr(), LA.data_ptr(), LB.data_ptr(), s.data_ptr(), p.bits, p.m, p.n,
                                     V.data_ptr(), Wq.data_ptr(), ws.data_ptr(), ws.numel(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream, kms, kl, kf)
    assert rc == 0 and int(st.item()) == 0
    assert kl[1] > 0 and kl[2] > 0 and kl[3] > 0 and kl[4] == 0, list(kl)
    check_against_oracle(p, V.cpu().numpy().astype(np.int64), Wq.cpu().numpy(), LA64, LB64, "wavefront profile")
