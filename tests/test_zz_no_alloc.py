"""The no-allocation solve, bakron_quantize_noalloc, called through the C ABI.

It exists for callers that cannot allocate device memory (a plugin whose
host application owns all of the GPU's memory, or a latency-critical path
that must not call cudaMalloc).  It must give the same codes as
bakron_quantize with a caller-provided workspace, also when called twice in
a row on different problems (the shared scratch keeps the previous call's
contents), and must refuse sizes beyond its fixed scratch.

The file name puts it last in collection order, so that a run stopping at
the first failure has run every other test before it.
"""

import ctypes

import numpy as np
import pytest

import oracle as O
from workloads import random_problem

pytestmark = pytest.mark.gpu

V_MATCH = 0.9999  # the parity bar of the other GPU tests
SCRATCH_BYTES = 80 << 20  # BAKRON_NOALLOC_SCRATCH_BYTES in bakron.h


@pytest.fixture(scope="module")
def env():
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import build as b

    b.build()
    lib = bk.load_library()
    torch.cuda.init()
    return bk, lib, torch


def _inputs(torch, p):
    LA64, LB64 = O.factors_of(p.A, p.B)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()  # noqa: E731
    s = None if p.scales is None else dev(p.scales)
    return dev(p.W), dev(LA64), dev(LB64), s


def _noalloc(lib, torch, W, LA, LB, s, bits):
    m, n = W.shape
    V = torch.empty((m, n), dtype=torch.int32, device="cuda")
    Wq = torch.empty((m, n), dtype=torch.float32, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.bakron_quantize_noalloc(W.data_ptr(), LA.data_ptr(), LB.data_ptr(), None if s is None else s.data_ptr(),
                                     bits, m, n, V.data_ptr(), Wq.data_ptr(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, V.cpu().numpy(), Wq.cpu().numpy(), int(st.item())


def test_noalloc_matches_workspace_entry_point_on_two_calls(env):
    bk, lib, torch = env
    # Two calls in a row: a larger problem first, then a smaller one, so the
    # second call runs on scratch full of the first call's state.
    for p in (random_problem(768, 896, bits=4, seed=8, w_std=0.02), random_problem(300, 170, bits=3, seed=4)):
        W, LA, LB, s = _inputs(torch, p)
        Vr, Wqr, str_ = bk.quantize(W, LA, LB, s, p.bits)
        torch.cuda.synchronize()
        assert int(str_.item()) == 0
        rc, Vn, Wqn, st = _noalloc(lib, torch, W, LA, LB, s, p.bits)
        assert rc == 0 and st == 0, (rc, st)
        Vr = Vr.cpu().numpy()
        assert O.match_fraction(Vn, Vr) >= V_MATCH
        assert np.array_equal(Vn, Vr) and np.array_equal(Wqn, Wqr.cpu().numpy())


@pytest.mark.parametrize("case", ["plain_rounding", "near_the_limit"])
def test_noalloc_matches_workspace_entry_point_edge_cases(env, case):
    """bits = 0 without scales (the alphabet Z of the 64 x 64 workload), and a
    1024 x 1024 layer whose solver state nearly fills the fixed scratch, so
    that its workspace layout reaches closest to the end of the array."""
    bk, lib, torch = env
    if case == "plain_rounding":
        p = random_problem(64, 64, bits=0, seed=21)
        assert p.scales is None
    else:
        p = random_problem(1024, 1024, bits=4, seed=22, w_std=0.02)
        assert SCRATCH_BYTES // 2 < bk.quantize_workspace_size(1024, 1024) <= SCRATCH_BYTES
    W, LA, LB, s = _inputs(torch, p)
    for _ in range(2):
        Vr, Wqr, str_ = bk.quantize(W, LA, LB, s, p.bits)
        torch.cuda.synchronize()
        assert int(str_.item()) == 0
        rc, Vn, Wqn, st = _noalloc(lib, torch, W, LA, LB, s, p.bits)
        assert rc == 0 and st == 0, (rc, st)
        assert np.array_equal(Vn, Vr.cpu().numpy()) and np.array_equal(Wqn, Wqr.cpu().numpy())


def test_noalloc_rejects_sizes_beyond_its_scratch(env):
    bk, lib, torch = env
    m, n = 2048, 2048  # 288 MiB of solver state
    assert bk.quantize_workspace_size(m, n) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x1000)
    rc = lib.bakron_quantize_noalloc(fake, fake, fake, None, 4, m, n, ctypes.c_void_p(0x2000),
                                     ctypes.c_void_p(0x3000), fake, None)
    assert rc == 4  # BAKRON_ERR_WORKSPACE, returned before anything is enqueued
    assert bk.quantize_workspace_size(1024, 1024) <= SCRATCH_BYTES
