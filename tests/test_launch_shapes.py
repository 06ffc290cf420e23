"""The decode GEMV's launch-shape chooser, checked on the host (no GPU):
tests/launch_shapes.cu includes the kernel header, enumerates every format,
M = 1..16, every lanes-per-row / rows-per-lane form the dispatcher uses and
a grid of K and N, and checks each shape's structure (power-of-two K parts
within their limits that cover K exactly, ring depth, thread count).  Shapes
that do not fit shared memory take the byte-wise kernel; this pins where
that happens: never at K <= 8192 (every decode shape of the workloads), at
K = 16384 only for M >= 8 (Q8_0 with two rows per lane from M = 8, where the
dispatcher first retries one row per lane; Q4_0 from M = 13 in the two-row
forms; both formats beyond that at larger K)."""
import os
import re
import shutil
import subprocess

import pytest

from block_quantized_matmul_gguf_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def report(tmp_path_factory):
    try:
        nvcc = build.nvcc_path()
    except RuntimeError:
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("shapes") / "launch_shapes")
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I", build.INCLUDE,
                    "-I", build.CSRC, "-o", exe, os.path.join(HERE, "launch_shapes.cu")],
                   check=True, capture_output=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    return r.returncode, r.stdout


def test_every_shape_is_well_formed(report):
    rc, out = report
    assert "violations 0" in out, [l for l in out.splitlines() if l.startswith("VIOLATION")][:10]
    assert rc == 0


def test_byte_wise_fallback_only_for_very_large_k(report):
    _, out = report
    refused = re.findall(r"^REFUSED (\w+) M=(\d+) L=(\d) R=(\d) k=(\d+) n=(\d+)", out, re.M)
    assert refused, "the enumeration reaches shapes that cannot fit (K up to 2^20)"
    for fmt, m, l, r, k, n in refused:
        k, m = int(k), int(m)
        assert k >= 16384, (fmt, m, l, r, k, n)
        if k == 16384:
            assert m >= 8, (fmt, m, l, r, k, n)
            if fmt == "q4_0":
                assert m >= 13 and r == "2", (fmt, m, l, r, k, n)


def test_row_pair_form_refused_only_for_large_k(report):
    """Q4_0 at M >= 11 leaves the row-pair form (for the per-block forms) only
    where a lane's K share would pass 1024 products (4 chunks per lane at two
    lanes a row: 8 chunks) or shared memory does not fit: K >= 16384, or a
    chunk count with an odd factor of 9 or more (K parts are powers of two).
    Never at the batched and decode workloads' sizes (K <= 8192)."""
    _, out = report
    refused = re.findall(r"ROWPAIR_REFUSED (\w+) M=(\d+) L=(\d) R=(\d) k=(\d+) n=(\d+)", out)
    for fmt, m, l, r, k, n in refused:
        chunks = int(k) // 256
        odd = chunks // (chunks & -chunks)
        assert fmt == "q4_0" and int(m) >= 11 and (int(k) >= 16384 or odd >= 9), (fmt, m, l, r, k, n)
    assert "ROWPAIR_REFUSED q4_0 M=16" in out  # K = 2^20 cannot fit
