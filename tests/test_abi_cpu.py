"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host -- no GPU needed (no compute call is made)."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "bakron.h")


@pytest.fixture(scope="module")
def lib():
    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import build as b

    b.build()
    return bk.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(bakron_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for need in ("bakron_prepare", "bakron_quantize", "bakron_factor", "bakron_quantize_host",
                 "bakron_status_string", "bakron_abi_version", "bakron_gptq_quantize",
                 "bakron_antidiag_quantize", "bakron_quantize_range", "bakron_quantize_scaled",
                 "bakron_row_scales", "bakron_pack_codes", "bakron_gram", "bakron_sq_norms", "bakron_damp",
                 "bakron_selftest_wait_timeout", "bakron_quantize_noalloc", "bakron_quantize_persistent",
                 "bakron_wavefront_plan_check"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    from kronecker_hessian_gptq_gb300 import _lib

    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings_and_version(lib):
    assert lib.bakron_abi_version() == 5
    assert lib.bakron_status_string(0) == b"BAKRON_OK"
    assert lib.bakron_status_string(4) == b"BAKRON_ERR_WORKSPACE"
    assert lib.bakron_status_string(99) == b"BAKRON_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    assert lib.bakron_quantize_workspace_size(0, 5) == 0
    assert lib.bakron_quantize_workspace_size(64, 64) >= 3 * 64 * 64 * 8
    q = lib.bakron_quantize_workspace_size(100, 37)
    assert lib.bakron_quantize_host_workspace_size(100, 37) > q
    assert lib.bakron_factor_workspace_size(0) == 0
    assert lib.bakron_prepare_workspace_size(10, 20) == max(
        lib.bakron_factor_workspace_size(10), lib.bakron_factor_workspace_size(20))


@pytest.mark.parametrize("entry", ["bakron_quantize", "bakron_quantize_persistent"])
def test_quantize_rejects_bad_arguments_before_any_launch(lib, entry):
    W = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    V, Wq = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    ws = ctypes.c_void_p(0x100000)
    big = lib.bakron_quantize_workspace_size(8, 8)
    q = getattr(lib, entry)
    assert q(W, W, W, None, 4, 0, 8, V, Wq, ws, big, W, None) == 1  # m < 1
    assert q(W, W, W, None, 4, 8, 0, V, Wq, ws, big, W, None) == 1  # n < 1
    for bits in (1, 9, -1, 16):
        assert q(W, W, W, None, bits, 8, 8, V, Wq, ws, big, W, None) == 1
    assert q(None, W, W, None, 4, 8, 8, V, Wq, ws, big, W, None) == 1  # null W
    assert q(W, W, W, None, 4, 8, 8, V, Wq, ws, big, None, None) == 1  # null status
    assert q(W, W, W, None, 4, 8, 8, V, W, ws, big, W, None) == 1  # Wq aliases W
    assert q(W, W, W, None, 4, 8, 8, V, V, ws, big, W, None) == 1  # Wq aliases V
    assert q(W, W, W, None, 4, 8, 8, V, Wq, ws, big - 1, W, None) == 4  # small workspace
    assert q(W, W, W, None, 4, 8, 8, V, Wq, None, big, W, None) == 4  # null workspace
    assert q(W, W, W, None, 4, 8, 8, V, Wq, ctypes.c_void_p(0x100010), big, W, None) == 4  # misaligned
    assert q(W, W, W, None, 4, 1 << 16, 1 << 16, V, Wq, ws, big, W, None) == 1  # m*n too large


def test_prepare_and_factor_reject_bad_arguments(lib):
    H = ctypes.c_void_p(0x1000)
    L = ctypes.c_void_p(0x2000)
    ws = ctypes.c_void_p(0x100000)
    assert lib.bakron_factor(H, 0, L, ws, 1 << 30, H, None) == 1
    assert lib.bakron_factor(H, 8, H, ws, 1 << 30, H, None) == 1  # H aliases Lhat
    assert lib.bakron_factor(H, 8, L, ws, 16, H, None) == 4
    assert lib.bakron_prepare(H, ctypes.c_void_p(0x1100), 0, 4, L, ctypes.c_void_p(0x3000), ws, 1 << 30, H,
                              None) == 1
    assert lib.bakron_prepare(H, ctypes.c_void_p(0x1100), 4, 4, L, L, ws, 1 << 30, H, None) == 1  # LA is LB


def test_python_binding_fails_loudly_without_library(tmp_path):
    from kronecker_hessian_gptq_gb300 import _lib

    saved = _lib._lib
    try:
        _lib._lib = None
        with pytest.raises(RuntimeError, match="libbakron.so not found"):
            _lib.load(str(tmp_path / "missing.so"))
    finally:
        _lib._lib = saved


def test_gptq_entry_point_rejects_bad_arguments(lib):
    W = ctypes.c_void_p(0x1000)
    V, Wq = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    ws = ctypes.c_void_p(0x100000)
    big = lib.bakron_gptq_workspace_size(8, 8)
    assert big == lib.bakron_quantize_workspace_size(8, 8)
    g = lib.bakron_gptq_quantize
    assert g(W, W, None, 4, 0, 8, V, Wq, ws, big, W, None) == 1  # m < 1
    assert g(None, W, None, 4, 8, 8, V, Wq, ws, big, W, None) == 1  # null W
    assert g(W, None, None, 4, 8, 8, V, Wq, ws, big, W, None) == 1  # null LA
    assert g(W, W, None, 9, 8, 8, V, Wq, ws, big, W, None) == 1  # bits
    assert g(W, W, None, 4, 8, 8, V, W, ws, big, W, None) == 1  # Wq aliases W
    assert g(W, W, None, 4, 8, 8, V, Wq, ws, big - 1, W, None) == 4  # small workspace


def test_range_scales_and_pack_entry_points_reject_bad_arguments(lib):
    W = ctypes.c_void_p(0x1000)
    V, Wq, S = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000)
    ws = ctypes.c_void_p(0x100000)
    big = lib.bakron_quantize_workspace_size(8, 8)
    q = lib.bakron_quantize_range
    assert q(W, W, None, None, -8, 7, 0, 8, V, Wq, ws, big, W, None) == 1  # m < 1
    assert q(W, None, None, None, -8, 7, 8, 8, V, Wq, ws, big, W, None) == 1  # null LA
    assert q(W, W, None, None, 7, -8, 8, 8, V, Wq, ws, big, W, None) == 1  # lo > hi
    assert q(W, W, None, None, 3, 3, 8, 8, V, Wq, ws, big, W, None) == 1  # lo == hi
    assert q(W, W, None, None, 1, 7, 8, 8, V, Wq, ws, big, W, None) == 1  # 0 not a code
    assert q(W, W, None, None, -40000, 7, 8, 8, V, Wq, ws, big, W, None) == 1  # |lo| too large
    assert q(W, W, None, None, -8, 7, 8, 8, V, V, ws, big, W, None) == 1  # V aliases Wq
    assert q(W, W, None, None, -8, 7, 8, 8, V, Wq, ws, big - 1, W, None) == 4  # small workspace
    r = lib.bakron_row_scales
    assert r(W, 0, 8, 0, -8, 7, 1, S, None) == 1  # m < 1
    assert r(W, 8, 8, -1, -8, 7, 1, S, None) == 1  # negative group
    assert r(W, 8, 8, 0, 0, 7, 1, S, None) == 1  # lo must be negative
    assert r(W, 8, 8, 0, -8, 0, 1, S, None) == 1  # hi must be positive
    assert r(W, 8, 8, 0, -8, 7, 0, S, None) == 1  # grid < 1
    assert r(W, 8, 8, 0, -8, 7, 257, S, None) == 1  # grid above the table
    assert r(W, 8, 8, 0, -8, 7, 4, W, None) == 1  # scales alias W
    assert r(None, 8, 8, 0, -8, 7, 4, S, None) == 1  # null W
    qs = lib.bakron_quantize_scaled
    assert qs(W, W, None, S, -1, None, -8, 7, 8, 8, V, Wq, ws, big, W, None) == 1  # negative group
    assert qs(W, W, None, S, 2, S, 7, -8, 8, 8, V, Wq, ws, big, W, None) == 1  # lo > hi
    assert qs(W, W, None, S, 2, S, -8, 7, 8, 8, W, Wq, ws, big, W, None) == 1  # V aliases W
    assert qs(W, W, None, S, 2, S, -8, 7, 8, 8, V, Wq, ws, big - 1, W, None) == 4  # small workspace
    p = lib.bakron_pack_codes
    assert p(V, 8, 8, 3, S, None) == 1  # bits not in {2, 4, 8}
    assert p(V, 8, 0, 4, S, None) == 1  # n < 1
    assert p(None, 8, 8, 4, S, None) == 1  # null V
    assert p(V, 8, 8, 4, None, None) == 1  # null out


def test_antidiag_entry_point_rejects_bad_arguments(lib):
    W = ctypes.c_void_p(0x1000)
    V, Wq = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    ws = ctypes.c_void_p(0x100000)
    need = lib.bakron_antidiag_workspace_size(8, 8)
    assert need == 512 + 256  # 8 x 8 double-float W~, two error rows (each padded to 256 bytes)
    assert lib.bakron_antidiag_workspace_size(0, 8) == 0
    a = lib.bakron_antidiag_quantize
    assert a(W, W, W, None, 4, 0, 8, V, Wq, ws, need, W, None) == 1  # m < 1
    assert a(W, W, None, None, 4, 8, 8, V, Wq, ws, need, W, None) == 1  # null LB
    assert a(W, W, W, None, 1, 8, 8, V, Wq, ws, need, W, None) == 1  # bits
    assert a(W, W, W, None, 4, 8, 8, V, V, ws, need, W, None) == 1  # V aliases Wq
    assert a(W, W, W, None, 4, 8, 8, V, Wq, ws, need - 1, W, None) == 4  # small workspace
    assert a(W, W, W, None, 4, 8, 8, V, Wq, ctypes.c_void_p(0x100010), need, W, None) == 4  # misaligned


def test_gram_entry_points_reject_bad_arguments(lib):
    X, G, st = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    w = ctypes.c_void_p(0x4000)
    ws = ctypes.c_void_p(0x100000)
    need = lib.bakron_gram_workspace_size(8, 8, 0)
    assert need == 16384 and lib.bakron_gram_workspace_size(8, 8, 1) == 3 * 16384  # one 128 x 64 block each
    assert lib.bakron_gram_workspace_size(129, 65, 0) == 4 * 16384
    g = lib.bakron_gram
    assert g(X, 0, 8, 8, None, 1.0, 0.0, G, ws, need, st, None) == 1  # d < 1
    assert g(X, 8, 0, 8, None, 1.0, 0.0, G, ws, need, st, None) == 1  # N < 1
    assert g(X, 8, 9, 8, None, 1.0, 0.0, G, ws, need, st, None) == 1  # ldx < N
    assert g(X, 8, 6, 6, None, 1.0, 0.0, G, ws, need, st, None) == 1  # ldx not a multiple of 8
    assert g(ctypes.c_void_p(0x1008), 8, 8, 8, None, 1.0, 0.0, G, ws, need, st, None) == 1  # X not 16-byte aligned
    assert g(X, 8, 8, 8, ctypes.c_void_p(0x4004), 1.0, 0.0, G, ws, need, st, None) == 1  # w not 16-byte aligned
    assert g(X, 8, 8, 8, w, 1.0, 0.0, X, ws, 3 * need, st, None) == 1  # G aliases X
    assert g(X, 8, 8, 8, w, 1.0, 0.0, G, ws, 3 * need, None, None) == 1  # no status word
    assert g(X, 8, 8, 8, w, 1.0, 0.0, G, ws, 3 * need - 1, st, None) == 4  # weighted needs three copies
    assert g(X, 8, 8, 8, None, 1.0, 0.0, G, ctypes.c_void_p(0x100010), need, st, None) == 4  # misaligned workspace
    assert lib.bakron_sq_norms(X, 4, 8, 7, w, None) == 1  # ldy < N
    assert lib.bakron_sq_norms(None, 4, 8, 8, w, None) == 1
    assert lib.bakron_damp(None, 4, 0.5, None) == 1
    assert lib.bakron_damp(G, 0, 0.5, None) == 1


def test_selftest_rejects_a_missing_status_word(lib):
    assert lib.bakron_selftest_wait_timeout(None, None) == 1


def test_workspace_holds_packed_factor_digits_only_on_large_layers(lib):
    """From 2^22 weights on the solve adds the factors' packed digits (10
    bytes per factor entry, 2 KB blocks of 32 rows x 32 columns x 5 digits
    per 128-column chunk)."""
    def packed(d):
        nch, nt = -(-d // 128), -(-d // 32)
        return -(-(nch * 4 * 5 * nt * 2048) // 256) * 256

    below = lib.bakron_quantize_workspace_size(2048, 2047)  # 2^22 - 2048 weights: digits made in the kernel
    at = lib.bakron_quantize_workspace_size(2048, 2048)  # 2^22 weights: packed digits for both factors
    assert at - below >= packed(2048) + packed(2048)
    assert lib.bakron_quantize_workspace_size(4104, 4096) > lib.bakron_quantize_workspace_size(4096, 4096)