"""The C-ABI library builds, loads and exports every entry point that
include/qmm.h declares; argument checks that return before any launch.
No kernel is launched here (these tests run without a GPU)."""
import ctypes
import os
import re

import pytest

from block_quantized_matmul_gguf_gb300 import build, qmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return qmm.load()


def test_header_declares_the_entry_points():
    syms = header_symbols()
    for name in ("qmm_dequant_q4_0", "qmm_dequant_q8_0", "qmm_gemv_q4_0", "qmm_gemv_q8_0",
                 "qmm_gemv_q4_0_multi", "qmm_gemv_q8_0_multi", "qmm_gemm_q4_0"):
        assert name in syms
    assert set(syms) <= set(qmm.EXPORTED) | set(syms)


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_compiles_on_its_own(tmp_path, lang, std):
    """A C or C++ caller includes the header and nothing else."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "qmm.h"\nint main(void) { return qmm_status_string(QMM_OK) == 0; }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(build.LIB_PATH)
    for name in header_symbols():
        assert hasattr(raw, name), name
    for name in qmm.EXPORTED:
        assert name in header_symbols(), name


def test_status_strings_and_version(lib):
    for s in range(8):
        assert qmm.status_string(s)
    assert "scratch" in qmm.status_string(qmm.QMM_ERR_SCRATCH)
    assert qmm.status_string(99) == "unknown status"
    assert qmm.qmm_version() >= 100


def test_copy_argument_checks(lib):
    """qmm_copy: nothing to copy is OK; a null pointer, overlapping ranges and
    pageable host memory (a kernel access to it would fault) are refused
    before any launch."""
    import numpy as np
    a = np.zeros(64, np.uint8)
    b = np.ones(64, np.uint8)
    L = lib
    assert L.qmm_copy(None, None, 0, None) == qmm.QMM_OK
    assert L.qmm_copy(None, b.ctypes.data, 16, None) == qmm.QMM_ERR_NULL
    assert L.qmm_copy(a.ctypes.data, None, 16, None) == qmm.QMM_ERR_NULL
    assert L.qmm_copy(b.ctypes.data + 8, b.ctypes.data, 16, None) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_copy(a.ctypes.data, b.ctypes.data, 64, None) == qmm.QMM_ERR_UNSUPPORTED
    assert (a == 0).all()


def test_null_and_shape_errors_return_before_any_launch(lib):
    L = lib
    assert L.qmm_gemv_q4_0(0, 16, 16, 1, 32, 64, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q4_0(16, 0, 16, 1, 32, 64, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q4_0(16, 16, 0, 1, 32, 64, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q8_0(16, 16, 4096, 0, 32, 64, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemv_q8_0(16, 16, 4096, 17, 32, 64, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemv_q4_0(16, 16, 4096, 1, 32, 48, 0) == qmm.QMM_ERR_SHAPE   # k % 32
    assert L.qmm_gemv_q4_0(16, 16, 4096, 1, 0, 64, 0) == qmm.QMM_ERR_SHAPE    # n = 0
    assert L.qmm_gemv_q4_0(16, 18, 4096, 1, 32, 64, 0) == qmm.QMM_ERR_ALIGN   # x % 4
    assert L.qmm_dequant_q4_0(0, 16, 4, 64, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_dequant_q8_0(16, 0, 4, 64, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_dequant_q8_0(16, 16, 4, 0, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_dequant_q4_0(16, 18, 4, 64, 0) == qmm.QMM_ERR_ALIGN
    assert L.qmm_gemm_q4_0(0, 16, 16, 256, 256, 256, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemm_q4_0(16, 16, 16, 0, 256, 256, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemm_q4_0(16, 16, 16, 256, 256, 288, 0) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_gemm_q4_0(18, 16, 16, 256, 256, 256, 0) == qmm.QMM_ERR_ALIGN


def test_overlapping_output_is_rejected(lib):
    # y overlapping w: rejected by the host check, nothing launched
    assert lib.qmm_gemv_q4_0(4096, 1 << 20, 4096 + 64, 1, 32, 64, 0) == qmm.QMM_ERR_UNSUPPORTED


def test_multi_argument_checks(lib):
    import ctypes
    Out = qmm.GemvOut
    arr = (Out * 2)()
    arr[0].w, arr[0].y, arr[0].n = 16, 4096, 32
    arr[1].w, arr[1].y, arr[1].n = 16, 0, 32
    assert lib.qmm_gemv_q4_0_multi(arr, 2, 16, 1, 64, 0) == qmm.QMM_ERR_NULL      # y NULL
    assert lib.qmm_gemv_q4_0_multi(arr, 0, 16, 1, 64, 0) == qmm.QMM_ERR_SHAPE     # count 0
    assert lib.qmm_gemv_q4_0_multi(arr, 5, 16, 1, 64, 0) == qmm.QMM_ERR_SHAPE     # count 5
    assert lib.qmm_gemv_q8_0_multi(None, 1, 16, 1, 64, 0) == qmm.QMM_ERR_NULL
    arr[1].y = 8192
    assert lib.qmm_gemv_q4_0_multi(arr, 2, 16, 1, 48, 0) == qmm.QMM_ERR_SHAPE     # k % 32
    assert lib.qmm_gemv_q4_0_multi(arr, 2, 16, 17, 64, 0) == qmm.QMM_ERR_SHAPE    # m


# ---- the entry points added for the fused FFN, Q8_0 prefill and workspaces ----
# (fake, never dereferenced pointer values: every case fails a check before any
# CUDA call; 1 << 24 apart so that ranges do not overlap unless meant to)

A, B, C, D, WS = 1 << 24, 2 << 24, 3 << 24, 4 << 24, 5 << 24


def test_geglu_gemv_argument_checks(lib):
    L = lib
    assert L.qmm_gemv_q4_0_geglu(0, B, C, D, 1, 64, 256, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q4_0_geglu(A, 0, C, D, 1, 64, 256, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q4_0_geglu(A, B, 0, D, 1, 64, 256, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q4_0_geglu(A, B, C, 0, 1, 64, 256, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemv_q4_0_geglu(A, B, C, D, 0, 64, 256, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemv_q4_0_geglu(A, B, C, D, 17, 64, 256, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemv_q4_0_geglu(A, B, C, D, 1, 64, 100, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemv_q4_0_geglu(A, B, C + 2, D, 1, 64, 256, 0) == qmm.QMM_ERR_ALIGN
    assert L.qmm_gemv_q4_0_geglu(A, B, C, C + 64, 1, 64, 256, 0) == qmm.QMM_ERR_UNSUPPORTED  # h over x
    assert L.qmm_gemv_q4_0_geglu(A, B, C, B + 16, 1, 64, 256, 0) == qmm.QMM_ERR_UNSUPPORTED  # h over wu


def test_q8_0_gemm_and_prefill_argument_checks(lib):
    L = lib
    for f in (L.qmm_gemm_q8_0, L.qmm_gemm_q4_0_prefill):
        assert f(0, B, C, 256, 256, 256, 0) == qmm.QMM_ERR_NULL
        assert f(A, 0, C, 256, 256, 256, 0) == qmm.QMM_ERR_NULL
        assert f(A, B, 0, 256, 256, 256, 0) == qmm.QMM_ERR_NULL
        assert f(A, B, C, 0, 256, 256, 0) == qmm.QMM_ERR_SHAPE
        assert f(A, B, C, 256, 256, 100, 0) == qmm.QMM_ERR_SHAPE
        assert f(A, B, C, 256, 256, 288, 0) == qmm.QMM_ERR_UNSUPPORTED   # k % 256
        assert f(A + 8, B, C, 256, 256, 256, 0) == qmm.QMM_ERR_ALIGN
        assert f(A, B + 8, C, 256, 256, 256, 0) == qmm.QMM_ERR_ALIGN
        assert f(A, B, C + 2, 256, 256, 256, 0) == qmm.QMM_ERR_ALIGN      # y % 4


@pytest.mark.parametrize("name", ["qmm_gemm_q4_0", "qmm_gemm_q8_0", "qmm_gemm_q4_0_prefill"])
def test_gemm_output_overlap_and_size_limits(lib, name):
    """y may overlap neither w nor x; m, n above 2^30 and k above 2^24 are
    valid shapes this build does not take.  All rejected before any launch."""
    f = getattr(lib, name)
    m, n, k = 256, 256, 256
    wbytes = n * (k // 32) * (18 if "q4_0" in name else 34)
    assert f(A, B, A + wbytes - 4, m, n, k, 0) == qmm.QMM_ERR_UNSUPPORTED   # y over w's tail
    assert f(A, B, B + 64, m, n, k, 0) == qmm.QMM_ERR_UNSUPPORTED           # y over x
    assert f(A, B, C, (1 << 30) + 1, 1, k, 0) == qmm.QMM_ERR_UNSUPPORTED
    assert f(A, B, C, 1, (1 << 30) + 1, k, 0) == qmm.QMM_ERR_UNSUPPORTED
    assert f(A, B, C, 1, 1, (1 << 24) + 256, 0) == qmm.QMM_ERR_UNSUPPORTED


def test_prefill_rejects_k_beyond_its_scratch(lib):
    """qmm_gemm_q4_0_prefill keeps one 256-row chunk of bf16 weights in its
    64 MiB scratch: k <= 131072.  Beyond that it returns QMM_ERR_SCRATCH
    before any CUDA call, whatever m is (the other GEMMs take such k)."""
    L = lib
    w, x, y = 1 << 24, 1 << 36, 1 << 40  # far apart: the large x does not reach y
    for m in (1, 300, 2048):
        assert L.qmm_gemm_q4_0_prefill(w, x, y, m, 4, 131072 + 256, 0) == qmm.QMM_ERR_SCRATCH
    assert L.qmm_gemm_q4_0_prefill(w, x, y, 1, 4, 1 << 24, 0) == qmm.QMM_ERR_SCRATCH
    # argument errors are still reported first
    assert L.qmm_gemm_q4_0_prefill(0, x, y, 1, 4, 131072 + 256, 0) == qmm.QMM_ERR_NULL


def test_geglu_gemm_argument_checks(lib):
    L = lib
    assert L.qmm_gemm_q4_0_geglu(0, B, C, D, 256, 64, 256, 0) == qmm.QMM_ERR_NULL
    assert L.qmm_gemm_q4_0_geglu(A, B, C, D, 0, 64, 256, 0) == qmm.QMM_ERR_SHAPE
    assert L.qmm_gemm_q4_0_geglu(A, B, C, D, 256, 64, 288, 0) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_gemm_q4_0_geglu(A, B + 8, C, D, 256, 64, 256, 0) == qmm.QMM_ERR_ALIGN
    assert L.qmm_gemm_q4_0_geglu(A, B, C, D + 1, 256, 64, 256, 0) == qmm.QMM_ERR_ALIGN
    assert L.qmm_gemm_q4_0_geglu(A, B, C, C + 256, 256, 64, 256, 0) == qmm.QMM_ERR_UNSUPPORTED


def test_workspace_sizes_and_checks(lib):
    assert qmm.qmm_gemm_workspace_bytes(8192, 2048) == 8192 * 2048 * 2
    assert qmm.qmm_gemm_workspace_bytes(100, 256) == 100 * 256 * 2
    assert qmm.qmm_gemm_workspace_bytes(0, 256) == 0
    # GeGLU: 128 rows (64 gate + 64 up) per 64 features
    assert qmm.qmm_gemm_workspace_bytes(100, 256, geglu=True) == 2 * 128 * 256 * 2
    assert qmm.qmm_gemm_workspace_bytes(8192, 2048, geglu=True) == 8192 * 2 * 2048 * 2
    L = lib
    m, n, k = 600, 256, 256  # m > 512: the two-phase path, so the workspace is checked
    need = n * k * 2
    for f in (L.qmm_gemm_q4_0_ws, L.qmm_gemm_q8_0_ws):
        assert f(A, B, C, m, n, k, WS, need - 1, 0) == qmm.QMM_ERR_SHAPE
        assert f(A, B, C, m, n, k, WS + 8, need, 0) == qmm.QMM_ERR_ALIGN
        assert f(A, B, C, m, n, k, C + 1024, need, 0) == qmm.QMM_ERR_UNSUPPORTED  # over y
        assert f(A, B, C, m, n, k, A, need, 0) == qmm.QMM_ERR_UNSUPPORTED         # over w
    gneed = qmm.qmm_gemm_workspace_bytes(n, k, geglu=True)
    g = L.qmm_gemm_q4_0_geglu_ws
    assert g(A, B, C, D, m, n, k, WS, gneed - 1, 0) == qmm.QMM_ERR_SHAPE
    assert g(A, B, C, D, m, n, k, WS + 8, gneed, 0) == qmm.QMM_ERR_ALIGN
    assert g(A, B, C, D, m, n, k, B, gneed, 0) == qmm.QMM_ERR_UNSUPPORTED           # over wu
