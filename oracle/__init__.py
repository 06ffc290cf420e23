"""CPU oracle for GGUF Q4_0 / Q8_0 block-quantized matrix products.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of what the
GPU library computes (dequantize each block exactly, accumulate in binary64).
Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import it.  It shares no code with the CUDA library and never imports it.

The C source is ``qmm_oracle.c``; this module compiles it with the host C
compiler (``-O2 -ffp-contract=off -fopenmp``, no fast-math) into
``oracle/_build/libqmm_oracle.so`` and wraps it with ctypes for numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_HDR = os.path.join(_HERE, "qmm_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libqmm_oracle.so")

Q4_0_BYTES = 18
Q8_0_BYTES = 34
QK = 32

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or stale."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= newest_src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["cc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.qmm_oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
    lib.qmm_oracle_fp16_to_f64.restype = ctypes.c_double
    lib.qmm_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.qmm_oracle_bf16_to_f64.restype = ctypes.c_double
    for name in ("qmm_oracle_dequant_q4_0", "qmm_oracle_dequant_q8_0"):
        getattr(lib, name).argtypes = [P, I64, I64, P]
        getattr(lib, name).restype = None
    for name in ("qmm_oracle_gemv_q4_0", "qmm_oracle_gemv_q8_0", "qmm_oracle_gemm_q4_0"):
        getattr(lib, name).argtypes = [P, P, I64, I64, I64, P, P]
        getattr(lib, name).restype = None
    for name in ("qmm_oracle_gemv_q4_0_at", "qmm_oracle_gemv_q8_0_at",
                 "qmm_oracle_gemm_q4_0_at"):
        getattr(lib, name).argtypes = [P, P, I64, P, P, I64, P, P]
        getattr(lib, name).restype = None
    lib.qmm_oracle_geglu_q4_0.argtypes = [P, P, P, I64, I64, I64, P, P, P, P, P]
    lib.qmm_oracle_geglu_q4_0.restype = None
    lib.qmm_oracle_geglu_q4_0_at.argtypes = [P, P, P, I64, P, P, I64, P, P, P, P, P]
    lib.qmm_oracle_geglu_q4_0_at.restype = None
    lib.qmm_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.qmm_oracle_set_threads.restype = None
    lib.qmm_oracle_get_threads.argtypes = []
    lib.qmm_oracle_get_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _blocks(w: np.ndarray, n: int, k: int, block_bytes: int) -> np.ndarray:
    if k % QK != 0 or k <= 0 or n <= 0:
        raise ValueError(f"bad shape n={n} k={k}")
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    if w.size != n * (k // QK) * block_bytes:
        raise ValueError(f"weight buffer has {w.size} bytes, expected "
                         f"{n * (k // QK) * block_bytes}")
    return w


def set_threads(n: int) -> None:
    _load().qmm_oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().qmm_oracle_get_threads())


def fp16_to_f64(h: int) -> float:
    return float(_load().qmm_oracle_fp16_to_f64(int(h) & 0xFFFF))


def bf16_to_f64(h: int) -> float:
    return float(_load().qmm_oracle_bf16_to_f64(int(h) & 0xFFFF))


def dequant_q4_0(w: np.ndarray, n: int, k: int) -> np.ndarray:
    """Dense binary32 [n][k] from Q4_0 blocks (exact)."""
    w = _blocks(w, n, k, Q4_0_BYTES)
    out = np.empty((n, k), dtype=np.float32)
    _load().qmm_oracle_dequant_q4_0(_ptr(w), n, k, _ptr(out))
    return out


def dequant_q8_0(w: np.ndarray, n: int, k: int) -> np.ndarray:
    """Dense binary32 [n][k] from Q8_0 blocks (exact)."""
    w = _blocks(w, n, k, Q8_0_BYTES)
    out = np.empty((n, k), dtype=np.float32)
    _load().qmm_oracle_dequant_q8_0(_ptr(w), n, k, _ptr(out))
    return out


def _product(name, w, x, m, n, k, block_bytes, x_dtype):
    w = _blocks(w, n, k, block_bytes)
    x = np.ascontiguousarray(x, dtype=x_dtype).reshape(-1)
    if x.size != m * k:
        raise ValueError(f"activation buffer has {x.size} values, expected {m * k}")
    y = np.empty((m, n), dtype=np.float64)
    bound = np.empty((m, n), dtype=np.float64)
    getattr(_load(), name)(_ptr(w), _ptr(x), m, n, k, _ptr(y), _ptr(bound))
    return y, bound


def gemv_q4_0(w, x, m, n, k):
    """(y, bound), each binary64 [m][n]: y = x . W^T with Q4_0 W, fp32 x."""
    return _product("qmm_oracle_gemv_q4_0", w, x, m, n, k, Q4_0_BYTES, np.float32)


def gemv_q8_0(w, x, m, n, k):
    """(y, bound), each binary64 [m][n]: y = x . W^T with Q8_0 W, fp32 x."""
    return _product("qmm_oracle_gemv_q8_0", w, x, m, n, k, Q8_0_BYTES, np.float32)


def gemm_q4_0(w, x_bf16_bits, m, n, k):
    """(y, bound) for bf16 X given as uint16 bit patterns [m][k]."""
    return _product("qmm_oracle_gemm_q4_0", w, x_bf16_bits, m, n, k, Q4_0_BYTES,
                    np.uint16)


def _product_at(name, w, x, m, n, k, mi, ni, block_bytes, x_dtype):
    w = _blocks(w, n, k, block_bytes)
    x = np.ascontiguousarray(x, dtype=x_dtype).reshape(-1)
    if x.size != m * k:
        raise ValueError(f"activation buffer has {x.size} values, expected {m * k}")
    mi = np.ascontiguousarray(mi, dtype=np.int64).reshape(-1)
    ni = np.ascontiguousarray(ni, dtype=np.int64).reshape(-1)
    if mi.shape != ni.shape:
        raise ValueError("index arrays differ in length")
    if mi.size and (mi.min() < 0 or mi.max() >= m or ni.min() < 0 or ni.max() >= n):
        raise ValueError("sample index out of range")
    y = np.empty(mi.size, dtype=np.float64)
    bound = np.empty(mi.size, dtype=np.float64)
    getattr(_load(), name)(_ptr(w), _ptr(x), k, _ptr(mi), _ptr(ni), mi.size,
                           _ptr(y), _ptr(bound))
    return y, bound


def gemv_q4_0_at(w, x, m, n, k, mi, ni):
    """Outputs (mi[i], ni[i]) of gemv_q4_0, with their bounds."""
    return _product_at("qmm_oracle_gemv_q4_0_at", w, x, m, n, k, mi, ni,
                       Q4_0_BYTES, np.float32)


def gemv_q8_0_at(w, x, m, n, k, mi, ni):
    return _product_at("qmm_oracle_gemv_q8_0_at", w, x, m, n, k, mi, ni,
                       Q8_0_BYTES, np.float32)


def gemm_q4_0_at(w, x_bf16_bits, m, n, k, mi, ni):
    return _product_at("qmm_oracle_gemm_q4_0_at", w, x_bf16_bits, m, n, k, mi, ni,
                       Q4_0_BYTES, np.uint16)


def geglu_q4_0(wg, wu, x, m, n, k):
    """(h, g, u, bound_g, bound_u), each binary64 [m][n]:
    g = x . Wg^T, u = x . Wu^T (Q4_0), h = gelu_tanh(g) * u."""
    wg = _blocks(wg, n, k, Q4_0_BYTES)
    wu = _blocks(wu, n, k, Q4_0_BYTES)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if x.size != m * k:
        raise ValueError(f"activation buffer has {x.size} values, expected {m * k}")
    outs = [np.empty((m, n), dtype=np.float64) for _ in range(5)]
    _load().qmm_oracle_geglu_q4_0(_ptr(wg), _ptr(wu), _ptr(x), m, n, k, *[_ptr(o) for o in outs])
    return tuple(outs)


def geglu_q4_0_at(wg, wu, x, m, n, k, mi, ni):
    """Outputs (mi[i], ni[i]) of geglu_q4_0: (h, g, u, bound_g, bound_u), each
    binary64 of the sample's length."""
    wg = _blocks(wg, n, k, Q4_0_BYTES)
    wu = _blocks(wu, n, k, Q4_0_BYTES)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if x.size != m * k:
        raise ValueError(f"activation buffer has {x.size} values, expected {m * k}")
    mi = np.ascontiguousarray(mi, dtype=np.int64).reshape(-1)
    ni = np.ascontiguousarray(ni, dtype=np.int64).reshape(-1)
    if mi.shape != ni.shape:
        raise ValueError("index arrays differ in length")
    if mi.size and (mi.min() < 0 or mi.max() >= m or ni.min() < 0 or ni.max() >= n):
        raise ValueError("sample index out of range")
    outs = [np.empty(mi.size, dtype=np.float64) for _ in range(5)]
    _load().qmm_oracle_geglu_q4_0_at(_ptr(wg), _ptr(wu), _ptr(x), k, _ptr(mi), _ptr(ni), mi.size,
                                     *[_ptr(o) for o in outs])
    return tuple(outs)
