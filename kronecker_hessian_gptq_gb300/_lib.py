"""ctypes loader for libbakron.so: signatures of the C ABI in include/bakron.h.

Loading fails loudly: there is no Python or CPU fallback for any entry point.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbakron.so")

OK = 0
STATUS_NAMES = {
    0: "BAKRON_OK",
    1: "BAKRON_ERR_INVALID_ARG",
    2: "BAKRON_ERR_NOT_SPD",
    3: "BAKRON_ERR_CUDA",
    4: "BAKRON_ERR_WORKSPACE",
    5: "BAKRON_ERR_TIMEOUT",
}
DEV_NONFINITE_W = 1
DEV_BAD_SCALE = 2
DEV_TIMEOUT = 4
KERNEL_CLASSES = ("setup", "tile_solve", "mid_push", "chunk_push", "sweep")

_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_int = ctypes.c_int
_vp = ctypes.c_void_p  # device or host pointers are passed as plain addresses

# name -> (restype, argtypes)
SIGNATURES = {
    "bakron_status_string": (ctypes.c_char_p, [_int]),
    "bakron_abi_version": (_int, []),
    "bakron_factor_workspace_size": (_sz, [_i64]),
    "bakron_factor": (_int, [_vp, _i64, _vp, _vp, _sz, _vp, _vp]),
    "bakron_prepare_workspace_size": (_sz, [_i64, _i64]),
    "bakron_prepare": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_quantize_workspace_size": (_sz, [_i64, _i64]),
    "bakron_quantize": (_int, [_vp, _vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_quantize_persistent": (_int, [_vp, _vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_gptq_workspace_size": (_sz, [_i64, _i64]),
    "bakron_gptq_quantize": (_int, [_vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_quantize_range": (_int, [_vp, _vp, _vp, _vp, _int, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_row_scales": (_int, [_vp, _i64, _i64, _i64, _int, _int, _int, _vp, _vp]),
    "bakron_quantize_scaled": (_int, [_vp, _vp, _vp, _vp, _i64, _vp, _int, _int, _i64, _i64, _vp, _vp, _vp, _sz,
                                      _vp, _vp]),
    "bakron_pack_codes": (_int, [_vp, _i64, _i64, _int, _vp, _vp]),
    "bakron_antidiag_workspace_size": (_sz, [_i64, _i64]),
    "bakron_antidiag_quantize": (_int, [_vp, _vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_gram_workspace_size": (_sz, [_i64, _i64, _int]),
    "bakron_gram": (_int, [_vp, _i64, _i64, _i64, _vp, ctypes.c_float, ctypes.c_float, _vp, _vp, _sz, _vp, _vp]),
    "bakron_sq_norms": (_int, [_vp, _i64, _i64, _i64, _vp, _vp]),
    "bakron_damp": (_int, [_vp, _i64, ctypes.c_float, _vp]),
    "bakron_selftest_wait_timeout": (_int, [_vp, _vp]),
    "bakron_quantize_profile": (_int, [_vp, _vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp,
                                        _vp, _vp, _vp]),
    "bakron_quantize_host_workspace_size": (_sz, [_i64, _i64]),
    "bakron_quantize_host": (_int, [_vp, _vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "bakron_quantize_noalloc": (_int, [_vp, _vp, _vp, _vp, _int, _i64, _i64, _vp, _vp, _vp, _vp]),
    "bakron_sweep_plan_check": (_int, [_i64, _i64, _vp]),
    "bakron_wavefront_plan_check": (_int, [_i64, _i64, _int, _int, _vp]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once and attach the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libbakron.so not found at {path}: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')"
        )
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, what: str) -> None:
    if status != OK:
        raise RuntimeError(f"{what} failed: {STATUS_NAMES.get(status, status)}")
