"""BaKron on GB300: Python binding of libbakron.so.

Thin argument marshalling over the C ABI declared in include/bakron.h: torch
is used only to allocate device memory and to name the current stream; every
step of the computation runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing, every call raises.

Source of the method: "BaKron: Efficient Quantization with Kronecker-Factored
Hessians" (arXiv 2608.06291), Sec. 3.

The calls, each a C ABI entry point of the same name with the prefix bakron_:
  factor, prepare        normalized inverse Cholesky factors L-hat (Sec. 3.2)
  quantize               the BaKron solve (Sec. 3.5, App. B eq. (2))
  quantize_persistent    the same solve as one persistent cooperative kernel
  quantize_host          the same from and to host memory
  gptq                   the one-sided case B = I (row-wise GPTQ, Sec. 1, Alg. 1)
  antidiag               BaKron-antidiagonal (Sec. 3.2, Alg. 3), the quartic baseline
  quantize_range         any integer alphabet {lo .. hi} (Sec. 3.1)
  quantize_scaled        per-run (group) and per-column scales (Sec. 3.1)
  row_scales             App. D scale choice with the MSE shrink search
  pack_codes             b-bit packed codes
  gram, sq_norms, damp   Kronecker factors from samples (Sec. 4.2, App. A.2, App. D)
"""

from __future__ import annotations

import ctypes
from typing import Optional, Tuple

from . import _lib

__all__ = [
    "load_library",
    "factor",
    "prepare",
    "quantize",
    "quantize_persistent",
    "quantize_host",
    "gptq",
    "antidiag",
    "gram",
    "sq_norms",
    "damp",
    "quantize_range",
    "quantize_scaled",
    "row_scales",
    "pack_codes",
    "quantize_workspace_size",
    "prepare_workspace_size",
]


def load_library():
    return _lib.load()


def _torch():
    import torch

    return torch


def _stream_handle(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _require_cuda_f32(t, shape, name):
    torch = _torch()
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == tuple(shape)):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {tuple(shape)}")


def _workspace(nbytes: int, device):
    torch = _torch()
    # torch's caching allocator hands out blocks aligned to at least 256 bytes
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def prepare_workspace_size(m: int, n: int) -> int:
    return int(_lib.load().bakron_prepare_workspace_size(m, n))


def quantize_workspace_size(m: int, n: int) -> int:
    return int(_lib.load().bakron_quantize_workspace_size(m, n))


def factor(H, ws=None, stream=None):
    """L-hat = Cholesky(H^-1) with unit-normalized columns (fp32, d x d).

    Returns (Lhat, info) where info is a 1-element int32 CUDA tensor: 0, or
    1 + the index of the first non-positive pivot met.
    """
    torch = _torch()
    lib = _lib.load()
    d = H.shape[0]
    _require_cuda_f32(H, (d, d), "H")
    L = torch.empty_like(H)
    info = torch.zeros(1, dtype=torch.int32, device=H.device)
    if ws is None:
        ws = _workspace(lib.bakron_factor_workspace_size(d), H.device)
    st = lib.bakron_factor(_ptr(H), d, _ptr(L), _ptr(ws), ws.numel(), _ptr(info), _stream_handle(stream))
    _lib.check(st, "bakron_factor")
    return L, info


def prepare(A, B, ws=None, stream=None):
    """(L-hat_A, L-hat_B, info[2]) for the input-side A (n x n) and output-side B (m x m)."""
    torch = _torch()
    lib = _lib.load()
    n, m = A.shape[0], B.shape[0]
    _require_cuda_f32(A, (n, n), "A")
    _require_cuda_f32(B, (m, m), "B")
    LA = torch.empty_like(A)
    LB = torch.empty_like(B)
    info = torch.zeros(2, dtype=torch.int32, device=A.device)
    if ws is None:
        ws = _workspace(lib.bakron_prepare_workspace_size(m, n), A.device)
    st = lib.bakron_prepare(_ptr(A), _ptr(B), m, n, _ptr(LA), _ptr(LB), _ptr(ws), ws.numel(), _ptr(info),
                            _stream_handle(stream))
    _lib.check(st, "bakron_prepare")
    return LA, LB, info


def quantize(W, LA, LB, scales=None, bits: int = 0, ws=None, out=None, stream=None):
    """BaKron quantization of W (m x n) given the normalized factors.

    Returns (V int32, Wq float32, status int32[1]) -- all CUDA tensors; the
    status word is 0 on success (BAKRON_DEV_* bits otherwise).
    """
    return _quantize("bakron_quantize", W, LA, LB, scales, bits, ws, out, stream)


def quantize_persistent(W, LA, LB, scales=None, bits: int = 0, ws=None, out=None, stream=None):
    """The same solve as quantize() as one persistent cooperative kernel
    (bakron_quantize_persistent); same arguments and results."""
    return _quantize("bakron_quantize_persistent", W, LA, LB, scales, bits, ws, out, stream)


def _quantize(entry, W, LA, LB, scales, bits, ws, out, stream):
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    _require_cuda_f32(W, (m, n), "W")
    _require_cuda_f32(LA, (n, n), "LA")
    _require_cuda_f32(LB, (m, m), "LB")
    if scales is not None:
        _require_cuda_f32(scales, (m,), "scales")
    if out is None:
        V = torch.empty((m, n), dtype=torch.int32, device=W.device)
        Wq = torch.empty((m, n), dtype=torch.float32, device=W.device)
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    else:
        V, Wq, status = out
    if ws is None:
        ws = _workspace(lib.bakron_quantize_workspace_size(m, n), W.device)
    st = getattr(lib, entry)(_ptr(W), _ptr(LA), _ptr(LB), _ptr(scales), int(bits), m, n, _ptr(V), _ptr(Wq),
                             _ptr(ws), ws.numel(), _ptr(status), _stream_handle(stream))
    _lib.check(st, entry)
    return V, Wq, status


def gptq(W, LA, scales=None, bits: int = 0, ws=None, out=None, stream=None):
    """Row-wise GPTQ of W (m x n): the one-sided case B = I of quantize()
    (bakron_gptq_quantize).  Returns (V, Wq, status) like quantize()."""
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    _require_cuda_f32(W, (m, n), "W")
    _require_cuda_f32(LA, (n, n), "LA")
    if scales is not None:
        _require_cuda_f32(scales, (m,), "scales")
    if out is None:
        V = torch.empty((m, n), dtype=torch.int32, device=W.device)
        Wq = torch.empty((m, n), dtype=torch.float32, device=W.device)
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    else:
        V, Wq, status = out
    if ws is None:
        ws = _workspace(lib.bakron_gptq_workspace_size(m, n), W.device)
    st = lib.bakron_gptq_quantize(_ptr(W), _ptr(LA), _ptr(scales), int(bits), m, n, _ptr(V), _ptr(Wq), _ptr(ws),
                                  ws.numel(), _ptr(status), _stream_handle(stream))
    _lib.check(st, "bakron_gptq_quantize")
    return V, Wq, status


def antidiag(W, LA, LB, scales=None, bits: int = 0, ws=None, out=None, stream=None):
    """BaKron-antidiagonal (Algorithm 3, bakron_antidiag_quantize): the same
    codes as quantize() by Theorem 3.2, with O(m^2 n^2) work in m + n - 1
    launches.  Returns (V, Wq, status) like quantize()."""
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    _require_cuda_f32(W, (m, n), "W")
    _require_cuda_f32(LA, (n, n), "LA")
    _require_cuda_f32(LB, (m, m), "LB")
    if scales is not None:
        _require_cuda_f32(scales, (m,), "scales")
    if out is None:
        V = torch.empty((m, n), dtype=torch.int32, device=W.device)
        Wq = torch.empty((m, n), dtype=torch.float32, device=W.device)
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    else:
        V, Wq, status = out
    if ws is None:
        ws = _workspace(lib.bakron_antidiag_workspace_size(m, n), W.device)
    st = lib.bakron_antidiag_quantize(_ptr(W), _ptr(LA), _ptr(LB), _ptr(scales), int(bits), m, n, _ptr(V), _ptr(Wq),
                                      _ptr(ws), ws.numel(), _ptr(status), _stream_handle(stream))
    _lib.check(st, "bakron_antidiag_quantize")
    return V, Wq, status


def _require_bf16_rows(X, name):
    torch = _torch()
    if not (X.is_cuda and X.dtype == torch.bfloat16 and X.dim() == 2 and X.stride(1) == 1):
        raise ValueError(f"{name} must be a 2-D bfloat16 CUDA tensor with contiguous rows")


def gram(X, w=None, alpha: Optional[float] = None, beta: float = 0.0, out=None, ws=None, stream=None):
    """G = beta G + alpha X diag(w) X^T for samples X (d x N bf16, feature-major)
    on the tensor cores (bakron_gram).  alpha defaults to 1/N (the sample
    mean).  Returns (G float32 d x d, status int32[1])."""
    torch = _torch()
    lib = _lib.load()
    _require_bf16_rows(X, "X")
    d, N = X.shape
    if w is not None:
        _require_cuda_f32(w, (N,), "w")
    G = torch.empty((d, d), dtype=torch.float32, device=X.device) if out is None else out
    _require_cuda_f32(G, (d, d), "G")
    status = torch.zeros(1, dtype=torch.int32, device=X.device)
    a = 1.0 / N if alpha is None else float(alpha)
    if ws is None:
        ws = _workspace(lib.bakron_gram_workspace_size(d, N, int(w is not None)), X.device)
    st = lib.bakron_gram(_ptr(X), d, N, X.stride(0), _ptr(w), a, float(beta), _ptr(G), _ptr(ws), ws.numel(),
                         _ptr(status), _stream_handle(stream))
    _lib.check(st, "bakron_gram")
    return G, status


def sq_norms(Y, out=None, stream=None):
    """|y_t|^2 of the columns of Y (m x N bf16): one Shampoo step's weights (bakron_sq_norms)."""
    torch = _torch()
    lib = _lib.load()
    _require_bf16_rows(Y, "Y")
    m, N = Y.shape
    w = torch.empty(N, dtype=torch.float32, device=Y.device) if out is None else out
    _require_cuda_f32(w, (N,), "w")
    st = lib.bakron_sq_norms(_ptr(Y), m, N, Y.stride(0), _ptr(w), _stream_handle(stream))
    _lib.check(st, "bakron_sq_norms")
    return w


def damp(G, rel: float = 0.5, stream=None):
    """G += rel * mean(diag G) * I in place (bakron_damp; App. D: rel = 0.5)."""
    lib = _lib.load()
    d = G.shape[0]
    _require_cuda_f32(G, (d, d), "G")
    st = lib.bakron_damp(_ptr(G), d, float(rel), _stream_handle(stream))
    _lib.check(st, "bakron_damp")
    return G


def quantize_range(W, LA, LB, scales, lo: int, hi: int, ws=None, out=None, stream=None):
    """BaKron (LB given) or row-wise GPTQ (LB None) over the integer alphabet
    {lo .. hi} (bakron_quantize_range).  Returns (V, Wq, status) like
    quantize()."""
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    _require_cuda_f32(W, (m, n), "W")
    _require_cuda_f32(LA, (n, n), "LA")
    if LB is not None:
        _require_cuda_f32(LB, (m, m), "LB")
    if scales is not None:
        _require_cuda_f32(scales, (m,), "scales")
    if out is None:
        V = torch.empty((m, n), dtype=torch.int32, device=W.device)
        Wq = torch.empty((m, n), dtype=torch.float32, device=W.device)
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    else:
        V, Wq, status = out
    if ws is None:
        ws = _workspace(lib.bakron_quantize_workspace_size(m, n), W.device)
    st = lib.bakron_quantize_range(_ptr(W), _ptr(LA), _ptr(LB), _ptr(scales), int(lo), int(hi), m, n, _ptr(V),
                                   _ptr(Wq), _ptr(ws), ws.numel(), _ptr(status), _stream_handle(stream))
    _lib.check(st, "bakron_quantize_range")
    return V, Wq, status


def row_scales(W, lo: int, hi: int, grid: int = 1, group: Optional[int] = None, out=None, stream=None):
    """Per-row scales of W for the alphabet {lo .. hi}, with a shrink search
    over `grid` factors from 1 down to 1/2 (bakron_row_scales).  Returns a
    float32 CUDA tensor of m scales, or of m x ceil(n / group) with a group
    size (one scale per run of `group` columns)."""
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    _require_cuda_f32(W, (m, n), "W")
    shape = (m,) if group is None else (m, -(-n // int(group)))
    scales = torch.empty(shape, dtype=torch.float32, device=W.device) if out is None else out
    _require_cuda_f32(scales, shape, "scales")
    st = lib.bakron_row_scales(_ptr(W), m, n, 0 if group is None else int(group), int(lo), int(hi), int(grid),
                               _ptr(scales), _stream_handle(stream))
    _lib.check(st, "bakron_row_scales")
    return scales


def quantize_scaled(W, LA, LB, scales, lo: int, hi: int, group: Optional[int] = None, col_scales=None, ws=None,
                    out=None, stream=None):
    """quantize_range() with one scale per entry, fp32(scales[i, j // group]
    * col_scales[j]) (bakron_quantize_scaled): `scales` holds m (group None)
    or m x ceil(n / group) run scales, or is None; `col_scales` n column
    scales or None.  Returns (V, Wq, status) like quantize()."""
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    _require_cuda_f32(W, (m, n), "W")
    _require_cuda_f32(LA, (n, n), "LA")
    if LB is not None:
        _require_cuda_f32(LB, (m, m), "LB")
    if scales is not None:
        _require_cuda_f32(scales, (m,) if group is None else (m, -(-n // int(group))), "scales")
    if col_scales is not None:
        _require_cuda_f32(col_scales, (n,), "col_scales")
    if out is None:
        V = torch.empty((m, n), dtype=torch.int32, device=W.device)
        Wq = torch.empty((m, n), dtype=torch.float32, device=W.device)
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    else:
        V, Wq, status = out
    if ws is None:
        ws = _workspace(lib.bakron_quantize_workspace_size(m, n), W.device)
    st = lib.bakron_quantize_scaled(_ptr(W), _ptr(LA), _ptr(LB), _ptr(scales), 0 if group is None else int(group),
                                    _ptr(col_scales), int(lo), int(hi), m, n, _ptr(V), _ptr(Wq), _ptr(ws), ws.numel(),
                                    _ptr(status), _stream_handle(stream))
    _lib.check(st, "bakron_quantize_scaled")
    return V, Wq, status


def pack_codes(V, bits: int, out=None, stream=None):
    """The codes V (int32, m x n) packed as bits-bit two's complement, rows
    byte-aligned (bakron_pack_codes).  Returns a uint8 CUDA tensor of
    m x ceil(n bits / 8)."""
    torch = _torch()
    lib = _lib.load()
    m, n = V.shape
    if not (V.is_cuda and V.dtype == torch.int32 and V.is_contiguous()):
        raise ValueError("V must be a contiguous int32 CUDA tensor")
    rowbytes = (n * int(bits) + 7) // 8
    P = torch.empty((m, rowbytes), dtype=torch.uint8, device=V.device) if out is None else out
    if not (P.is_cuda and P.dtype == torch.uint8 and P.is_contiguous() and tuple(P.shape) == (m, rowbytes)):
        raise ValueError("out must be a contiguous uint8 CUDA tensor of m x ceil(n bits / 8)")
    st = lib.bakron_pack_codes(_ptr(V), m, n, int(bits), _ptr(P), _stream_handle(stream))
    _lib.check(st, "bakron_pack_codes")
    return P


def quantize_host(W, LA, LB, scales=None, bits: int = 0, dev_ws=None, out=None, stream=None) -> Tuple:
    """Same as quantize() from and to HOST (CPU, ideally pinned) torch tensors.

    The library copies the inputs to the device workspace, solves, copies V
    and Wq back and synchronizes.  Returns (V, Wq, status:int).
    """
    torch = _torch()
    lib = _lib.load()
    m, n = W.shape
    for t, shp, name in ((W, (m, n), "W"), (LA, (n, n), "LA"), (LB, (m, m), "LB")):
        if t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"{name} must be a contiguous float32 CPU tensor of shape {shp}")
    if out is None:
        V = torch.empty((m, n), dtype=torch.int32, pin_memory=True)
        Wq = torch.empty((m, n), dtype=torch.float32, pin_memory=True)
    else:
        V, Wq = out
    if dev_ws is None:
        dev_ws = _workspace(lib.bakron_quantize_host_workspace_size(m, n), torch.device("cuda"))
    status = ctypes.c_int32(0)
    st = lib.bakron_quantize_host(_ptr(W), _ptr(LA), _ptr(LB), _ptr(scales), int(bits), m, n, _ptr(V), _ptr(Wq),
                                  _ptr(dev_ws), dev_ws.numel(), ctypes.addressof(status), _stream_handle(stream))
    _lib.check(st, "bakron_quantize_host")
    return V, Wq, int(status.value)
