"""The persistent sweep's task plan, checked on the host (no GPU) through the
C ABI: every delayed update the sweep's bands do not apply themselves is
carried by exactly one tensor-core task ("BaKron: Efficient Quantization with
Kronecker-Factored Hessians", App. B eq. (1): the updates of finished
entries form one product L_B E L_A^T restricted to the later entries), and
in the ideal schedule each task's sources are complete well before its
first target is needed."""

import ctypes

import pytest

SHAPES = [(1, 1), (1, 9), (9, 1), (31, 33), (64, 64), (65, 97), (100, 37), (130, 70), (200, 600), (300, 170),
          (768, 896), (1000, 1300), (1300, 1000), (1024, 1024), (4100, 4100)]


@pytest.fixture(scope="module")
def lib():
    import kronecker_hessian_gptq_gb300 as bk

    return bk.load_library()


@pytest.mark.parametrize("m,n", SHAPES)
def test_plan_covers_every_delayed_update_once(lib, m, n):
    st = (ctypes.c_int64 * 3)()
    rc = lib.bakron_sweep_plan_check(m, n, st)
    assert rc == 0 and st[2] == 0, (rc, list(st))
    if st[0]:
        assert st[1] >= 32, list(st)  # steps between sources complete and first target needed


def test_plan_rejects_bad_sizes(lib):
    st = (ctypes.c_int64 * 3)()
    assert lib.bakron_sweep_plan_check(0, 5, st) == 1  # BAKRON_ERR_INVALID_ARG
    assert lib.bakron_sweep_plan_check(5, 5, None) == 1
