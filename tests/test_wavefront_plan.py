"""The tile wavefront's launch schedule (bakron_quantize, and
bakron_gptq_quantize with L_B = I), checked on the host (no GPU) through the
C ABI: every delayed update -- the terms of the product L_B E L_A^T
restricted to the later entries ("BaKron: Efficient Quantization with
Kronecker-Factored Hessians", App. B eq. (1)), split along tile columns
(column terms) and tile rows (row terms) -- is carried exactly once, by a
target's own solve, a mid push or a chunk product, and each is complete by
the step whose solve waits for it."""

import ctypes

import pytest

SHAPES = [(1, 1), (1, 9), (9, 1), (31, 33), (64, 64), (65, 97), (100, 37), (130, 70), (200, 600), (300, 170),
          (768, 896), (1000, 1300), (1300, 1000), (1024, 1024), (2100, 2100), (4096, 4096), (4100, 4100),
          (4096, 1024), (1024, 4096)]
LAG = 5  # B + 1: the solve of step K waits for the chunk products launched at step K - 5


@pytest.fixture(scope="module")
def lib():
    import kronecker_hessian_gptq_gb300 as bk

    return bk.load_library()


def _check(lib, m, n, colpush, lag=LAG):
    st = (ctypes.c_int64 * 3)()
    rc = lib.bakron_wavefront_plan_check(m, n, colpush, lag, st)
    return rc, list(st)


@pytest.mark.parametrize("m,n", SHAPES)
@pytest.mark.parametrize("colpush", [1, 0])
def test_schedule_carries_every_delayed_update_once_and_in_time(lib, m, n, colpush):
    rc, st = _check(lib, m, n, colpush)
    assert rc == 0 and st[2] == 0, (rc, st)
    if st[1] >= 0:
        assert st[1] == LAG, st  # the nearest chunk target is solved exactly when the solve waits


def test_a_longer_lag_than_the_schedule_gives_is_caught(lib):
    """Planted mistake: claiming that the solves wait six steps for the chunk
    products (the schedule gives five) must report late targets."""
    rc, st = _check(lib, 1024, 1024, 1, lag=LAG + 1)
    assert rc == 1 and st[2] > 0, (rc, st)


def test_plan_check_rejects_bad_arguments(lib):
    st = (ctypes.c_int64 * 3)()
    assert lib.bakron_wavefront_plan_check(0, 5, 1, LAG, st) == 1  # BAKRON_ERR_INVALID_ARG
    assert lib.bakron_wavefront_plan_check(5, 5, 2, LAG, st) == 1
    assert lib.bakron_wavefront_plan_check(5, 5, 1, 0, st) == 1
    assert lib.bakron_wavefront_plan_check(5, 5, 1, LAG, None) == 1
    assert lib.bakron_wavefront_plan_check(1 << 16, 5, 1, LAG, st) == 1
