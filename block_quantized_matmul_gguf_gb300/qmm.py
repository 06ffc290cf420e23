"""Thin ctypes binding of libqmm.so (include/qmm.h), same entry-point names.

Only argument marshalling happens here: tensors become device pointers and
the stream becomes the current torch CUDA stream unless one is given.  Every
step of the computation runs in the library's CUDA kernels.  There is no
fallback: if libqmm.so cannot be loaded, every call raises.

Each function takes torch CUDA tensors (or raw integer device pointers) and
raises :class:`QmmError` when the library returns a non-OK status.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

QMM_OK = 0
QMM_ERR_NULL = 1
QMM_ERR_SHAPE = 2
QMM_ERR_ALIGN = 3
QMM_ERR_UNSUPPORTED = 4
QMM_ERR_CUDA = 5
QMM_ERR_TIMEOUT = 6
QMM_ERR_SCRATCH = 7
QMM_GEMV_MAX_M = 16

QMM_GEMV_MAX_OUTPUTS = 4

EXPORTED = (
    "qmm_dequant_q4_0", "qmm_dequant_q8_0", "qmm_gemv_q4_0", "qmm_gemv_q8_0",
    "qmm_gemv_q4_0_multi", "qmm_gemv_q8_0_multi", "qmm_gemv_q4_0_geglu", "qmm_gemv_q4_0_tc",
    "qmm_gemm_q4_0", "qmm_gemm_q8_0", "qmm_gemm_q4_0_geglu",
    "qmm_gemm_q4_0_ws", "qmm_gemm_q8_0_ws", "qmm_gemm_q4_0_geglu_ws", "qmm_gemm_q4_0_prefill",
    "qmm_gemm_workspace_bytes", "qmm_gemm_geglu_workspace_bytes", "qmm_status_string", "qmm_version", "qmm_get_device_error",
    "qmm_set_wait_timeout_ns", "qmm_selftest_wait_timeout", "qmm_copy",
)


class GemvOut(ctypes.Structure):
    """struct qmm_gemv_out: one weight matrix and its output."""
    _fields_ = [("w", ctypes.c_void_p), ("y", ctypes.c_void_p), ("n", ctypes.c_int64)]


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libqmm.so (building it first if asked and it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        if not build_if_missing:
            raise OSError(f"libqmm.so not built at {path}")
        _build.build_library()
    lib = ctypes.CDLL(path)
    P, I64, I32, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
    SZ = ctypes.c_size_t
    sig = {
        "qmm_dequant_q4_0": [P, P, I64, I64, P],
        "qmm_dequant_q8_0": [P, P, I64, I64, P],
        "qmm_gemv_q4_0": [P, P, P, I32, I64, I64, P],
        "qmm_gemv_q8_0": [P, P, P, I32, I64, I64, P],
        "qmm_gemv_q4_0_tc": [P, P, P, I32, I64, I64, P],
        "qmm_gemm_q4_0": [P, P, P, I64, I64, I64, P],
        "qmm_gemm_q8_0": [P, P, P, I64, I64, I64, P],
        "qmm_gemv_q4_0_geglu": [P, P, P, P, I32, I64, I64, P],
        "qmm_gemm_q4_0_geglu": [P, P, P, P, I64, I64, I64, P],
        "qmm_gemm_q4_0_ws": [P, P, P, I64, I64, I64, P, SZ, P],
        "qmm_gemm_q4_0_prefill": [P, P, P, I64, I64, I64, P],
        "qmm_gemm_q8_0_ws": [P, P, P, I64, I64, I64, P, SZ, P],
        "qmm_gemm_q4_0_geglu_ws": [P, P, P, P, I64, I64, I64, P, SZ, P],
        "qmm_gemv_q4_0_multi": [ctypes.POINTER(GemvOut), I32, P, I32, I64, P],
        "qmm_gemv_q8_0_multi": [ctypes.POINTER(GemvOut), I32, P, I32, I64, P],
        "qmm_get_device_error": [P],
        "qmm_selftest_wait_timeout": [U64, P],
        "qmm_copy": [P, P, SZ, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.qmm_status_string.argtypes = [ctypes.c_int]
    lib.qmm_status_string.restype = ctypes.c_char_p
    lib.qmm_version.argtypes = []
    lib.qmm_version.restype = ctypes.c_int
    for name in ("qmm_gemm_workspace_bytes", "qmm_gemm_geglu_workspace_bytes"):
        getattr(lib, name).argtypes = [I64, I64]
        getattr(lib, name).restype = SZ
    lib.qmm_set_wait_timeout_ns.argtypes = [U64]
    lib.qmm_set_wait_timeout_ns.restype = None
    _lib = lib
    return lib


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != QMM_OK:
        raise QmmError(status, where)


def status_string(status: int) -> str:
    return load().qmm_status_string(int(status)).decode()


def qmm_version() -> int:
    return int(load().qmm_version())


def qmm_dequant_q4_0(w, out, n: int, k: int, stream=None) -> None:
    _check(load().qmm_dequant_q4_0(_ptr(w), _ptr(out), n, k, _stream(stream)),
           "qmm_dequant_q4_0")


def qmm_dequant_q8_0(w, out, n: int, k: int, stream=None) -> None:
    _check(load().qmm_dequant_q8_0(_ptr(w), _ptr(out), n, k, _stream(stream)),
           "qmm_dequant_q8_0")


def _ptr_pinned_ok(t) -> int:
    """Like _ptr, but a page-locked host tensor is accepted too."""
    if t is None or isinstance(t, int) or t.is_cuda:
        return _ptr(t)
    if not t.is_pinned():
        raise ValueError("host tensor must be page-locked (pin_memory())")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def qmm_copy(dst, src, nbytes: int, stream=None) -> None:
    """Stream-ordered copy by the SMs; dst and src are device memory or
    page-locked host memory."""
    _check(load().qmm_copy(_ptr_pinned_ok(dst), _ptr_pinned_ok(src), int(nbytes),
                           _stream(stream)), "qmm_copy")


def qmm_gemv_q4_0(w, x, y, m: int, n: int, k: int, stream=None) -> None:
    _check(load().qmm_gemv_q4_0(_ptr(w), _ptr(x), _ptr(y), m, n, k, _stream(stream)),
           "qmm_gemv_q4_0")


def qmm_gemv_q8_0(w, x, y, m: int, n: int, k: int, stream=None) -> None:
    _check(load().qmm_gemv_q8_0(_ptr(w), _ptr(x), _ptr(y), m, n, k, _stream(stream)),
           "qmm_gemv_q8_0")


def qmm_gemv_q4_0_tc(w, x, y, m: int, n: int, k: int, stream=None) -> None:
    """The Q4_0 GEMV on the tensor cores (batched decode, same accuracy bound)."""
    _check(load().qmm_gemv_q4_0_tc(_ptr(w), _ptr(x), _ptr(y), m, n, k, _stream(stream)),
           "qmm_gemv_q4_0_tc")


def _outs(outs):
    arr = (GemvOut * max(1, len(outs)))()
    for i, (w, y, n) in enumerate(outs):
        arr[i].w = _ptr(w)
        arr[i].y = _ptr(y)
        arr[i].n = int(n)
    return arr


def qmm_gemv_q4_0_multi(outs, x, m: int, k: int, stream=None) -> None:
    """outs: sequence of (w, y, n) sharing the activations x [m][k]."""
    _check(load().qmm_gemv_q4_0_multi(_outs(outs), len(outs), _ptr(x), m, k, _stream(stream)),
           "qmm_gemv_q4_0_multi")


def qmm_gemv_q8_0_multi(outs, x, m: int, k: int, stream=None) -> None:
    _check(load().qmm_gemv_q8_0_multi(_outs(outs), len(outs), _ptr(x), m, k, _stream(stream)),
           "qmm_gemv_q8_0_multi")


def qmm_gemv_q4_0_geglu(wg, wu, x, h, m: int, n: int, k: int, stream=None) -> None:
    """h[m][n] = gelu_tanh(x . wg^T) * (x . wu^T), one launch."""
    _check(load().qmm_gemv_q4_0_geglu(_ptr(wg), _ptr(wu), _ptr(x), _ptr(h), m, n, k,
                                      _stream(stream)), "qmm_gemv_q4_0_geglu")


def qmm_gemm_q4_0(w, x_bf16, y, m: int, n: int, k: int, stream=None) -> None:
    _check(load().qmm_gemm_q4_0(_ptr(w), _ptr(x_bf16), _ptr(y), m, n, k, _stream(stream)),
           "qmm_gemm_q4_0")


def qmm_gemm_q8_0(w, x_bf16, y, m: int, n: int, k: int, stream=None) -> None:
    _check(load().qmm_gemm_q8_0(_ptr(w), _ptr(x_bf16), _ptr(y), m, n, k, _stream(stream)),
           "qmm_gemm_q8_0")


def qmm_gemm_q4_0_geglu(wg, wu, x_bf16, h_bf16, m: int, n: int, k: int, stream=None) -> None:
    """h (bf16) = gelu_tanh(X . wg^T) * (X . wu^T) on the tensor cores, one launch."""
    _check(load().qmm_gemm_q4_0_geglu(_ptr(wg), _ptr(wu), _ptr(x_bf16), _ptr(h_bf16), m, n, k,
                                      _stream(stream)), "qmm_gemm_q4_0_geglu")


def qmm_gemm_workspace_bytes(n: int, k: int, geglu: bool = False) -> int:
    lib = load()
    return int((lib.qmm_gemm_geglu_workspace_bytes if geglu else lib.qmm_gemm_workspace_bytes)(n, k))


def qmm_gemm_q4_0_ws(w, x_bf16, y, m, n, k, ws, ws_bytes, stream=None) -> None:
    _check(load().qmm_gemm_q4_0_ws(_ptr(w), _ptr(x_bf16), _ptr(y), m, n, k, _ptr(ws), int(ws_bytes),
                                   _stream(stream)), "qmm_gemm_q4_0_ws")


def qmm_gemm_q8_0_ws(w, x_bf16, y, m, n, k, ws, ws_bytes, stream=None) -> None:
    _check(load().qmm_gemm_q8_0_ws(_ptr(w), _ptr(x_bf16), _ptr(y), m, n, k, _ptr(ws), int(ws_bytes),
                                   _stream(stream)), "qmm_gemm_q8_0_ws")


def qmm_gemm_q4_0_geglu_ws(wg, wu, x_bf16, h_bf16, m, n, k, ws, ws_bytes, stream=None) -> None:
    _check(load().qmm_gemm_q4_0_geglu_ws(_ptr(wg), _ptr(wu), _ptr(x_bf16), _ptr(h_bf16), m, n, k,
                                         _ptr(ws), int(ws_bytes), _stream(stream)),
           "qmm_gemm_q4_0_geglu_ws")


def qmm_gemm_q4_0_prefill(w, x_bf16, y, m: int, n: int, k: int, stream=None) -> None:
    """The Q4_0 prefill product without a workspace argument, for callers
    that cannot allocate device memory: long prompts run in two phases on a
    64 MiB scratch array owned by the library (k <= 131072, else status
    QMM_ERR_SCRATCH).  Calls that overlap on the GPU race on that scratch."""
    _check(load().qmm_gemm_q4_0_prefill(_ptr(w), _ptr(x_bf16), _ptr(y), m, n, k, _stream(stream)),
           "qmm_gemm_q4_0_prefill")


def qmm_get_device_error(stream=None) -> int:
    """Synchronise `stream`; return (and clear) the device error word."""
    return int(load().qmm_get_device_error(_stream(stream)))


def qmm_set_wait_timeout_ns(ns: int) -> None:
    load().qmm_set_wait_timeout_ns(int(ns))


def qmm_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(load().qmm_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "qmm_selftest_wait_timeout")


# ---- tensor-level conveniences (allocate the output, then call the ABI) ----

def dequant(fmt: str, w, n: int, k: int, stream=None):
    import torch
    out = torch.empty((n, k), dtype=torch.float32, device=w.device)
    (qmm_dequant_q4_0 if fmt == "q4_0" else qmm_dequant_q8_0)(w, out, n, k, stream)
    return out


def gemv(fmt: str, w, x, n: int, k: int, stream=None):
    import torch
    m = x.shape[0]
    y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    (qmm_gemv_q4_0 if fmt == "q4_0" else qmm_gemv_q8_0)(w, x, y, m, n, k, stream)
    return y


def gemv_tc_q4_0(w, x, n: int, k: int, stream=None):
    import torch
    m = x.shape[0]
    y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    qmm_gemv_q4_0_tc(w, x, y, m, n, k, stream)
    return y


def geglu_q4_0(wg, wu, x, n: int, k: int, stream=None):
    import torch
    m = x.shape[0]
    h = torch.empty((m, n), dtype=torch.float32, device=x.device)
    qmm_gemv_q4_0_geglu(wg, wu, x, h, m, n, k, stream)
    return h


def gemm(fmt: str, w, x_bf16, n: int, k: int, stream=None, workspace=None):
    """workspace: a device tensor of at least qmm_gemm_workspace_bytes(n, k) bytes
    (the two-phase path for m > 256), or None (the fused call)."""
    import torch
    m = x_bf16.shape[0]
    y = torch.empty((m, n), dtype=torch.float32, device=x_bf16.device)
    if workspace is None:
        (qmm_gemm_q4_0 if fmt == "q4_0" else qmm_gemm_q8_0)(w, x_bf16, y, m, n, k, stream)
    else:
        (qmm_gemm_q4_0_ws if fmt == "q4_0" else qmm_gemm_q8_0_ws)(
            w, x_bf16, y, m, n, k, workspace, workspace.numel() * workspace.element_size(), stream)
    return y


def gemm_geglu_q4_0(wg, wu, x_bf16, n: int, k: int, stream=None, workspace=None):
    """Returns h as an int16 tensor of bf16 bit patterns [m][n]."""
    import torch
    m = x_bf16.shape[0]
    h = torch.empty((m, n), dtype=torch.int16, device=x_bf16.device)
    if workspace is None:
        qmm_gemm_q4_0_geglu(wg, wu, x_bf16, h, m, n, k, stream)
    else:
        qmm_gemm_q4_0_geglu_ws(wg, wu, x_bf16, h, m, n, k, workspace,
                               workspace.numel() * workspace.element_size(), stream)
    return h


def gemm_q4_0(w, x_bf16, n: int, k: int, stream=None):
    import torch
    m = x_bf16.shape[0]
    y = torch.empty((m, n), dtype=torch.float32, device=x_bf16.device)
    qmm_gemm_q4_0(w, x_bf16, y, m, n, k, stream)
    return y
