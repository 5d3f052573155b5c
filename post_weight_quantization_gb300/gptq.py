"""Python binding of the GPTQ C ABI (include/gptq.h).

Argument marshalling only: every step of the path runs in the CUDA library
``libgptq.so``. PyTorch provides device memory and the current stream. The
functions keep the C names; they take torch tensors, check dtype/device/shape,
allocate outputs and workspaces with torch when the caller passes none, and raise
``GPTQError`` on a non-OK status.

If the library has not been built, importing this module fails with an ImportError
that says how to build it; there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgptq.so")

GPTQ_OK = 0
GPTQ_ERR_INVALID_ARG = 1
GPTQ_ERR_NOT_PD = 2
GPTQ_ERR_NONFINITE = 3
GPTQ_ERR_UNSUPPORTED = 4
GPTQ_ERR_CUDA = 5
GPTQ_ERR_TIMEOUT = 6
GPTQ_WS_FACTOR = 0
GPTQ_WS_QUANTIZE = 1
GPTQ_WS_DEQUANT_GEMM = 2

_c_int, _c_i64, _c_size, _c_float, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/gptq.h
SIGNATURES = {
    "gptq_status_string": (ctypes.c_char_p, [_c_int]),
    "gptq_last_error": (ctypes.c_char_p, []),
    "gptq_version": (_c_int, []),
    "gptq_launch_count": (ctypes.c_uint64, []),
    "gptq_device_check": (_c_int, [_vp]),
    "gptq_hessian_accumulate": (_c_int, [_vp, _c_i64, _c_i64, _c_i64, _vp, _c_i64, _c_float, _c_int, _vp]),
    "gptq_workspace_size": (_c_size, [_c_int, _c_i64, _c_i64, _c_int, _c_int, _c_int]),
    "gptq_factor": (_c_int, [_vp, _c_i64, _c_float, _c_int, _vp, _vp, _vp, _c_size, ctypes.POINTER(_c_i64), _vp]),
    "gptq_factor_status": (_c_int, [_vp, ctypes.POINTER(_c_i64), _vp]),
    "gptq_factor_static": (_c_int, [_vp, _c_i64, _c_float, _c_int, _vp, _vp, ctypes.POINTER(_c_i64), _vp]),
    "gptq_quantize_layer": (_c_int, [_vp, _c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp,
                                     _vp, _vp, _vp, _c_size, ctypes.POINTER(_c_i64), _vp]),
    "gptq_unpack_codes": (_c_int, [_vp, _c_i64, _c_i64, _c_int, _vp, _vp]),
    "gptq_dequant_gemv": (_c_int, [_vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_int, _vp, _c_i64, _c_i64, _vp, _c_i64,
                                   _vp]),
    "gptq_gemm_f32": (_c_int, [_c_int, _c_int, _c_int, _c_i64, _c_i64, _c_i64, _vp, _c_i64, _vp, _c_i64, _vp, _c_i64,
                               _c_float, _c_float, _c_int, _vp]),
    "gptq_wait_selftest": (_c_int, [_c_int, _c_i64, _vp]),
    "gptq_dequant_gemm": (_c_int, [_vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_int, _vp, _c_i64, _c_i64, _vp, _c_int,
                                   _c_i64, _vp, _c_size, _vp]),
    "gptq_pipeline_create": (_c_int, [_c_i64, _c_i64, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_i64,
                                      ctypes.POINTER(_vp)]),
    "gptq_pipeline_run": (_c_int, [_vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "gptq_pipeline_status": (_c_int, [_vp, ctypes.POINTER(_c_i64), _vp]),
    "gptq_pipeline_destroy": (_c_int, [_vp]),
}


class GPTQError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(message)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m post_weight_quantization_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _check(status: int, what: str) -> None:
    if status != GPTQ_OK:
        name = _lib.gptq_status_string(status).decode()
        detail = _lib.gptq_last_error().decode()
        raise GPTQError(status, f"{what}: {name}: {detail}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need_cuda(t: torch.Tensor, name: str, dtypes) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")


def _need_buffer(t: torch.Tensor, name: str, shape, dtypes) -> None:
    """A tensor the library reads or writes as a dense array: CUDA, one of `dtypes`, the
    exact `shape`, contiguous."""
    _need_cuda(t, name, dtypes)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_rows(t: torch.Tensor, name: str, rows: int, cols: int, dtypes) -> None:
    """A contiguous row-major array of `cols` columns with at least `rows` rows (the
    library reads the first `rows`)."""
    _need_cuda(t, name, dtypes)
    if t.dim() != 2 or t.shape[1] != cols or t.shape[0] < rows:
        raise ValueError(f"{name} must have shape (>= {rows}, {cols}), got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _one_device(*tensors) -> torch.device:
    """The common device of the tensors, which must be the current CUDA device (the
    library launches on the current device)."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one device, got {sorted(map(str, devs))}")
    dev = devs.pop()
    if dev.index is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {dev} but the current device is cuda:{torch.cuda.current_device()}; "
                         f"call under torch.cuda.device({dev.index})")
    return dev


def _need_workspace(ws: torch.Tensor, nbytes: int) -> int:
    """Bytes of a caller workspace (any dtype), which must cover `nbytes`."""
    _need_cuda(ws, "ws", (torch.uint8, torch.int8, torch.int32, torch.float32, torch.int64, torch.float64))
    if not ws.is_contiguous():
        raise ValueError("ws must be contiguous")
    have = ws.numel() * ws.element_size()
    if have < nbytes:
        raise ValueError(f"ws holds {have} bytes, {nbytes} are needed")
    return have


# ----------------------------------------------------------------------------------
def gptq_status_string(status: int) -> str:
    return _lib.gptq_status_string(status).decode()


def gptq_last_error() -> str:
    return _lib.gptq_last_error().decode()


def gptq_version() -> int:
    return _lib.gptq_version()


def gptq_launch_count() -> int:
    return int(_lib.gptq_launch_count())


def gptq_device_check(stream=None) -> None:
    _check(_lib.gptq_device_check(_stream(stream)), "gptq_device_check")


def gptq_wait_selftest(which: int, limit_ns: int = 1_000_000, stream=None) -> int:
    """Run one of the library's bounded waits alone on something that never completes
    (which 0: the panels' counter wait, 1: the mbarrier wait) with a short limit; returns
    the status (GPTQ_ERR_TIMEOUT is the expected outcome) without raising."""
    return int(_lib.gptq_wait_selftest(int(which), int(limit_ns), _stream(stream)))


def gptq_workspace_size(which: int, m: int, d: int, bits: int = 4, group_size: int = 128,
                        blocksize: int = 128) -> int:
    return int(_lib.gptq_workspace_size(which, m, d, bits, group_size, blocksize))


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's allocator returns 512-byte aligned blocks, above the 256 bytes the ABI needs
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def gptq_hessian_accumulate(X: torch.Tensor, H: torch.Tensor, alpha: float = 2.0, zero_first: bool = False,
                            stream=None) -> torch.Tensor:
    """H[i, j] (i <= j) = (0 if zero_first else H[i, j]) + alpha * sum_t X[t, i] X[t, j].

    X: (n, d) bf16 (or its uint16 bits) on the GPU, row stride a multiple of 8.
    H: (d, d) float32 on the GPU; only the upper triangle is written.
    """
    _need_cuda(X, "X", (torch.bfloat16, torch.uint16, torch.int16))
    _need_cuda(H, "H", (torch.float32,))
    if X.dim() != 2 or H.dim() != 2 or X.stride(1) != 1 or H.stride(1) != 1:
        raise ValueError("X and H must be 2-D with unit column stride")
    n, d = X.shape
    if H.shape[0] != d or H.shape[1] != d:
        raise ValueError("H must be d x d")
    _one_device(X, H)
    _check(_lib.gptq_hessian_accumulate(_ptr(X), n, d, X.stride(0), _ptr(H), H.stride(0), float(alpha),
                                        int(bool(zero_first)), _stream(stream)), "gptq_hessian_accumulate")
    return H


def gptq_factor(H: torch.Tensor, percdamp: float = 0.01, act_order: bool = False,
                Hinv1: Optional[torch.Tensor] = None, perm_out: Optional[torch.Tensor] = None,
                ws: Optional[torch.Tensor] = None, sync: bool = True, stream=None):
    """Damp H, optionally compute the act-order permutation, and return (Hinv1, perm, info).

    With sync=True the call waits for the GPU and raises GPTQError on a failed
    factorization (info holds the failing column); otherwise info is None.
    """
    _need_cuda(H, "H", (torch.float32,))
    d = H.shape[0]
    if H.dim() != 2 or H.shape[1] != d or not H.is_contiguous():
        raise ValueError("H must be a contiguous d x d tensor")
    dev = H.device
    if Hinv1 is None:
        Hinv1 = torch.empty((d, d), dtype=torch.float32, device=dev)
    _need_buffer(Hinv1, "Hinv1", (d, d), (torch.float32,))
    if act_order:
        if perm_out is None:
            perm_out = torch.empty(d, dtype=torch.int32, device=dev)
        _need_buffer(perm_out, "perm_out", (d,), (torch.int32,))
    need = gptq_workspace_size(GPTQ_WS_FACTOR, 0, d)
    if ws is None:
        ws = _workspace(need, dev)
    ws_bytes = _need_workspace(ws, need)
    _one_device(H, Hinv1, perm_out if act_order else None, ws)
    info = _c_i64(-1)
    st = _lib.gptq_factor(_ptr(H), d, float(percdamp), int(bool(act_order)), _ptr(perm_out) if act_order else None,
                          _ptr(Hinv1), _ptr(ws), ws_bytes, ctypes.byref(info) if sync else None, _stream(stream))
    _check(st, "gptq_factor")
    return Hinv1, (perm_out if act_order else None), (int(info.value) if sync else None)


def gptq_factor_static(H: torch.Tensor, Hinv1: torch.Tensor, percdamp: float = 0.01, act_order: bool = False,
                       perm_out: Optional[torch.Tensor] = None, stream=None):
    """gptq_factor with the library's own device scratch (d <= 2048) instead of a workspace,
    for callers that cannot allocate device memory. Outputs must be passed in. The call
    always waits for the GPU (its outcome is read back from the shared scratch) and
    raises GPTQError on a failed factorization."""
    _need_cuda(H, "H", (torch.float32,))
    _need_cuda(Hinv1, "Hinv1", (torch.float32,))
    d = H.shape[0]
    if not H.is_contiguous() or not Hinv1.is_contiguous() or Hinv1.shape != H.shape:
        raise ValueError("H and Hinv1 must be contiguous d x d tensors")
    if act_order:
        _need_buffer(perm_out, "perm_out", (d,), (torch.int32,))
    _one_device(H, Hinv1, perm_out if act_order else None)
    info = _c_i64(-1)
    st = _lib.gptq_factor_static(_ptr(H), d, float(percdamp), int(bool(act_order)),
                                 _ptr(perm_out) if act_order else None, _ptr(Hinv1), ctypes.byref(info),
                                 _stream(stream))
    _check(st, "gptq_factor_static")
    return Hinv1, (perm_out if act_order else None), int(info.value)


@dataclass
class QuantizedLayer:
    qweight: torch.Tensor      # (m, ceil(d * bits / 32)) int32 words (uint32 bit patterns)
    scales: torch.Tensor       # (m, G) float32
    zeros: torch.Tensor        # (m, G) float32
    col_losses: torch.Tensor   # (d,) float32
    bits: int
    group_size: int
    d: int


def gptq_quantize_layer(W: torch.Tensor, Hinv1: torch.Tensor, perm: Optional[torch.Tensor] = None, bits: int = 4,
                        group_size: int = 128, blocksize: int = 128, out: Optional[QuantizedLayer] = None,
                        ws: Optional[torch.Tensor] = None, sync: bool = False, stream=None) -> QuantizedLayer:
    """Run the blocked GPTQ column loop on W (m x d, fp32 or bf16) with Hinv1 from gptq_factor."""
    _need_cuda(W, "W", (torch.float32, torch.bfloat16))
    _need_cuda(Hinv1, "Hinv1", (torch.float32,))
    if W.dim() != 2 or W.stride(1) != 1:
        raise ValueError("W must be 2-D with unit column stride")
    m, d = W.shape
    if Hinv1.shape != (d, d) or not Hinv1.is_contiguous():
        raise ValueError("Hinv1 must be a contiguous d x d tensor")
    if perm is not None:
        _need_buffer(perm, "perm", (d,), (torch.int32,))
    dev = W.device
    G = 1 if group_size == -1 else (d // group_size if group_size > 0 else 1)
    if out is None:
        out = QuantizedLayer(
            qweight=torch.empty((m, (d * bits + 31) // 32), dtype=torch.int32, device=dev),
            scales=torch.empty((m, G), dtype=torch.float32, device=dev),
            zeros=torch.empty((m, G), dtype=torch.float32, device=dev),
            col_losses=torch.empty(d, dtype=torch.float32, device=dev),
            bits=bits, group_size=group_size, d=d)
    if (out.bits, out.group_size, out.d) != (bits, group_size, d):
        raise ValueError(f"out describes bits={out.bits}, group_size={out.group_size}, d={out.d}; "
                         f"the call has {bits}, {group_size}, {d}")
    _need_buffer(out.qweight, "out.qweight", (m, (d * bits + 31) // 32), (torch.int32,))
    _need_buffer(out.scales, "out.scales", (m, G), (torch.float32,))
    _need_buffer(out.zeros, "out.zeros", (m, G), (torch.float32,))
    _need_buffer(out.col_losses, "out.col_losses", (d,), (torch.float32,))
    need = gptq_workspace_size(GPTQ_WS_QUANTIZE, m, d, bits, group_size, blocksize)
    if ws is None:
        ws = _workspace(need, dev)
    ws_bytes = _need_workspace(ws, need)
    _one_device(W, Hinv1, perm, out.qweight, out.scales, out.zeros, out.col_losses, ws)
    info = _c_i64(0)
    st = _lib.gptq_quantize_layer(_ptr(W), 0 if W.dtype == torch.float32 else 1, m, d, W.stride(0), _ptr(Hinv1),
                                  _ptr(perm), bits, group_size, blocksize, _ptr(out.qweight), _ptr(out.scales),
                                  _ptr(out.zeros), _ptr(out.col_losses), _ptr(ws), ws_bytes,
                                  ctypes.byref(info) if sync else None, _stream(stream))
    _check(st, "gptq_quantize_layer")
    return out


def gptq_unpack_codes(qweight: torch.Tensor, m: int, d: int, bits: int, stream=None) -> torch.Tensor:
    _need_rows(qweight, "qweight", m, (d * bits + 31) // 32, (torch.int32,))
    _one_device(qweight)
    codes = torch.empty((m, d), dtype=torch.uint8, device=qweight.device)
    _check(_lib.gptq_unpack_codes(_ptr(qweight), m, d, bits, _ptr(codes), _stream(stream)), "gptq_unpack_codes")
    return codes


def gptq_dequant_gemv(q: "QuantizedLayer", X: torch.Tensor, m: int, g_idx: Optional[torch.Tensor] = None,
                      Y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Y = X W_hat^T (T x m, fp32) from the packed layer q and bf16 tokens X (T x d)."""
    _need_cuda(X, "X", (torch.bfloat16, torch.int16))
    if X.dim() != 2 or X.stride(1) != 1 or X.shape[1] != q.d:
        raise ValueError("X must be T x d with unit column stride")
    G = 1 if q.group_size == -1 else (q.d // q.group_size if q.group_size > 0 else 1)
    _need_rows(q.qweight, "q.qweight", m, (q.d * q.bits + 31) // 32, (torch.int32,))
    _need_rows(q.scales, "q.scales", m, G, (torch.float32,))
    _need_rows(q.zeros, "q.zeros", m, G, (torch.float32,))
    if g_idx is not None:
        _need_buffer(g_idx, "g_idx", (q.d,), (torch.int32,))
    T = X.shape[0]
    if Y is None:
        Y = torch.empty((T, m), dtype=torch.float32, device=X.device)
    _need_cuda(Y, "Y", (torch.float32,))
    if Y.dim() != 2 or tuple(Y.shape) != (T, m) or Y.stride(1) != 1:
        raise ValueError(f"Y must be ({T}, {m}) with unit column stride, got {tuple(Y.shape)}")
    _one_device(q.qweight, q.scales, q.zeros, g_idx, X, Y)
    st = _lib.gptq_dequant_gemv(_ptr(q.qweight), _ptr(q.scales), _ptr(q.zeros), _ptr(g_idx), m, q.d, q.bits,
                                q.group_size, _ptr(X), T, X.stride(0), _ptr(Y), Y.stride(0), _stream(stream))
    _check(st, "gptq_dequant_gemv")
    return Y


def gptq_dequant_gemm(q: "QuantizedLayer", X: torch.Tensor, m: int, Y: Optional[torch.Tensor] = None,
                      out_bf16: bool = False, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Y = X W_hat^T (T x m) on the tensor cores from the packed layer q and bf16 tokens X
    (T x d); fp32 output, or bf16 with out_bf16 (the next layer's calibration inputs)."""
    _need_cuda(X, "X", (torch.bfloat16, torch.int16))
    if X.dim() != 2 or X.stride(1) != 1 or X.shape[1] != q.d:
        raise ValueError("X must be T x d with unit column stride")
    G = 1 if q.group_size == -1 else (q.d // q.group_size if q.group_size > 0 else 1)
    _need_rows(q.qweight, "q.qweight", m, (q.d * q.bits + 31) // 32, (torch.int32,))
    _need_rows(q.scales, "q.scales", m, G, (torch.float32,))
    _need_rows(q.zeros, "q.zeros", m, G, (torch.float32,))
    T = X.shape[0]
    ydt = torch.bfloat16 if out_bf16 else torch.float32
    if Y is None:
        Y = torch.empty((T, m), dtype=ydt, device=X.device)
    _need_cuda(Y, "Y", (ydt,))
    if Y.dim() != 2 or tuple(Y.shape) != (T, m) or Y.stride(1) != 1:
        raise ValueError(f"Y must be ({T}, {m}) with unit column stride, got {tuple(Y.shape)}")
    need = gptq_workspace_size(GPTQ_WS_DEQUANT_GEMM, m, q.d)
    if ws is None:
        ws = _workspace(need, X.device)
    ws_bytes = _need_workspace(ws, need)
    _one_device(q.qweight, q.scales, q.zeros, X, Y, ws)
    st = _lib.gptq_dequant_gemm(_ptr(q.qweight), _ptr(q.scales), _ptr(q.zeros), m, q.d, q.bits, q.group_size,
                                _ptr(X), T, X.stride(0), _ptr(Y), int(bool(out_bf16)), Y.stride(0), _ptr(ws), ws_bytes,
                                _stream(stream))
    _check(st, "gptq_dequant_gemm")
    return Y


def gptq_gemm_f32(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, a_kmajor: bool, b_kmajor: bool,
                  alpha: float = 1.0, beta: float = 0.0, engine: int = 0, lower_tiles: bool = False,
                  stream=None) -> torch.Tensor:
    """C = beta C + alpha A B with the library's block-update GEMM (test helper).

    a_kmajor: A is stored (M, K) row-major, else (K, M); b_kmajor: B is stored (N, K),
    else (K, N). C is (M, N)."""
    for t, nm in ((A, "A"), (B, "B"), (C, "C")):
        _need_cuda(t, nm, (torch.float32,))
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{nm} must be 2-D with unit column stride")
    M, N = C.shape
    K = A.shape[1] if a_kmajor else A.shape[0]
    if (A.shape[0] if a_kmajor else A.shape[1]) != M:
        raise ValueError(f"A must be ({M}, K) when a_kmajor, else (K, {M}); got {tuple(A.shape)}")
    if tuple(B.shape) != ((N, K) if b_kmajor else (K, N)):
        raise ValueError(f"B must be {(N, K) if b_kmajor else (K, N)}, got {tuple(B.shape)}")
    _one_device(A, B, C)
    _check(_lib.gptq_gemm_f32(engine, int(a_kmajor), int(b_kmajor), M, N, K, _ptr(A), A.stride(0), _ptr(B),
                              B.stride(0), _ptr(C), C.stride(0), float(alpha), float(beta), int(lower_tiles),
                              _stream(stream)), "gptq_gemm_f32")
    return C


# ----------------------------------------------------------------------------------
def quantize_layer(W: torch.Tensor, X_batches, bits: int = 4, group_size: int = 128, blocksize: int = 128,
                   percdamp: float = 0.01, act_order: bool = False, alpha: float = 2.0, stream=None):
    """The whole per-layer path: H from calibration batches, Hinv1, then the column loop.

    Returns (QuantizedLayer, H, Hinv1, perm).
    """
    d = W.shape[1]
    H = torch.empty((d, d), dtype=torch.float32, device=W.device)
    first = True
    for X in X_batches:
        gptq_hessian_accumulate(X, H, alpha=alpha, zero_first=first, stream=stream)
        first = False
    if first:
        raise ValueError("no calibration batch")
    Hinv1, perm, _ = gptq_factor(H, percdamp=percdamp, act_order=act_order, stream=stream)
    q = gptq_quantize_layer(W, Hinv1, perm, bits=bits, group_size=group_size, blocksize=blocksize, stream=stream)
    return q, H, Hinv1, perm


def sequential_quantize(X0: torch.Tensor, weights, bits: int = 4, group_size: int = 128, blocksize: int = 128,
                        percdamp: float = 0.01, act_order: bool = False, alpha: float = 2.0, stream=None):
    """Layers quantized one after another ("The GPTQ Algorithm", procedure steps 1-4): each
    layer of a chain of linear layers is calibrated on the bf16 outputs of the quantized
    layers before it. X0 (n x d0, bf16) are the first layer's inputs; weights[l] is
    (m_l x d_l) with d_{l+1} = m_l. Layer l is quantized from its inputs, then
    gptq_dequant_gemm computes its outputs from the packed layer, rounded to bf16, which
    become layer l+1's inputs.

    Returns (layers, inputs, output): layers[l] = (QuantizedLayer, perm), inputs[l] the
    bf16 tokens layer l was calibrated on, output the last layer's bf16 outputs."""
    X = X0
    layers, inputs = [], []
    for W in weights:
        if X.shape[1] != W.shape[1]:
            raise ValueError(f"a layer of width {W.shape[1]} follows outputs of width {X.shape[1]}")
        inputs.append(X)
        q, _, _, perm = quantize_layer(W, [X], bits=bits, group_size=group_size, blocksize=blocksize,
                                       percdamp=percdamp, act_order=act_order, alpha=alpha, stream=stream)
        layers.append((q, perm))
        X = gptq_dequant_gemm(q, X, W.shape[0], out_bf16=True, stream=stream)
    return layers, inputs, X


def _host_empty(shape, dtype) -> torch.Tensor:
    """A host buffer for the pipeline's copies: page-locked where CUDA is present (so the
    copies run asynchronously), ordinary memory otherwise."""
    return torch.empty(shape, dtype=dtype, pin_memory=torch.cuda.is_available())


def _on_device(dev: torch.device):
    return torch.cuda.device(dev) if torch.cuda.is_available() else contextlib.nullcontext()


class HostPipeline:
    """End-to-end quantization of one layer from host buffers, over the library's native
    pipeline (gptq_pipeline_create / _run / _status / _destroy).

    The library streams the calibration tokens to the GPU in chunks on its own copy
    stream while the Hessian accumulates the chunk before on the caller's stream (two
    device chunk buffers in turn), copies W, runs the factor and the column loop, and
    copies the packed codes, scales, zeros, per-column losses (and the act-order
    permutation) back into the pinned host tensors held here. Its device memory is one
    allocation made at construction and reused by every run.
    """

    def __init__(self, m: int, d: int, bits: int = 4, group_size: int = 128, blocksize: int = 128,
                 percdamp: float = 0.01, act_order: bool = False, chunk_tokens: int = 32768,
                 w_dtype=torch.bfloat16, device="cuda"):
        if w_dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("w_dtype must be torch.float32 or torch.bfloat16")
        self.m, self.d, self.bits, self.group_size, self.blocksize = m, d, bits, group_size, blocksize
        self.percdamp, self.act_order, self.chunk, self.w_dtype = percdamp, act_order, chunk_tokens, w_dtype
        self.device = torch.device(device)
        self._h = None
        h = _vp()
        with _on_device(self.device):
            _check(_lib.gptq_pipeline_create(m, d, 1 if w_dtype == torch.bfloat16 else 0, bits, group_size, blocksize,
                                             float(percdamp), 1 if act_order else 0, chunk_tokens, ctypes.byref(h)),
                   "gptq_pipeline_create")
        self._h = h
        G = 1 if group_size == -1 else d // group_size
        self.host_out = QuantizedLayer(
            qweight=_host_empty((m, (d * bits + 31) // 32), torch.int32), scales=_host_empty((m, G), torch.float32),
            zeros=_host_empty((m, G), torch.float32), col_losses=_host_empty((d,), torch.float32),
            bits=bits, group_size=group_size, d=d)
        self.perm = _host_empty((d,), torch.int32) if act_order else None

    def __del__(self):
        if getattr(self, "_h", None) is not None:
            _lib.gptq_pipeline_destroy(self._h)
            self._h = None

    def bytes_h2d(self, n_tokens: int) -> int:
        return n_tokens * self.d * 2 + self.m * self.d * (2 if self.w_dtype == torch.bfloat16 else 4)

    def bytes_d2h(self) -> int:
        o = self.host_out
        n = sum(t.numel() * t.element_size() for t in (o.qweight, o.scales, o.zeros, o.col_losses))
        return n + (self.d * 4 if self.act_order else 0)

    def run(self, W_host: torch.Tensor, X_host: torch.Tensor, stream=None) -> QuantizedLayer:
        """W_host (m x d host tensor of the pipeline's dtype), X_host (n x d bf16 bits as
        int16, host); both row-major with unit column stride (any row stride), pinned
        for the copies to overlap the Hessian. Returns the host output tensors; they
        are complete once the stream has been synchronized (check() reads the outcome)."""
        for t, name in ((W_host, "W_host"), (X_host, "X_host")):
            if t.is_cuda or t.dim() != 2 or t.shape[1] != self.d or t.stride(1) != 1:
                raise ValueError(f"{name} must be a host tensor (rows, {self.d}) with unit column stride")
        if W_host.dtype != self.w_dtype or W_host.shape[0] != self.m:
            raise ValueError(f"W_host must be ({self.m}, {self.d}) {self.w_dtype}")
        if X_host.dtype not in (torch.int16, torch.bfloat16):
            raise TypeError("X_host must hold bf16 bits (torch.int16 or torch.bfloat16)")
        o = self.host_out
        with _on_device(self.device):
            _check(_lib.gptq_pipeline_run(self._h, W_host.data_ptr(), W_host.stride(0), X_host.data_ptr(),
                                          X_host.shape[0], X_host.stride(0), o.qweight.data_ptr(),
                                          o.scales.data_ptr(), o.zeros.data_ptr(), o.col_losses.data_ptr(),
                                          _ptr(self.perm), _stream(stream)), "gptq_pipeline_run")
        return o

    def check(self, stream=None) -> int:
        """Synchronize the stream and raise GPTQError if the last run's factor or column
        loop failed; returns info (-1 on success)."""
        info = _c_i64(0)
        with _on_device(self.device):
            _check(_lib.gptq_pipeline_status(self._h, ctypes.byref(info), _stream(stream)), "gptq_pipeline_status")
        return int(info.value)
