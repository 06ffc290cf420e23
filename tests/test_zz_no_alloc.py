"""The workspace-free prefill GEMM, qmm_gemm_q4_0_prefill, against the entry
point it stands in for, qmm_gemm_q4_0_ws (the same two-phase product with a
caller-allocated workspace).

qmm_gemm_q4_0_prefill serves callers that cannot allocate device memory: a
host whose device memory all belongs to its own allocator (a serving arena or
a framework's caching allocator with a fixed budget) and which forbids a
library's cudaMalloc, or a plugin interface that hands an operator its inputs
and outputs only, with no workspace slot.  It runs on a 64 MiB scratch array
that the library itself holds on each GPU, so every call shares that array
and finds the previous call's data in it.

The test makes two calls in a row with different data and shapes (the second
one in three column chunks, at the largest K the scratch takes) and checks
each output against the workspace entry point's output within the GEMM
tolerance of the other tests (and bit for bit, since both run the same
kernels), with the tolerance scale from the CPU oracle.  It also checks that
the second call leaves the device's free memory unchanged.

This file is named so that pytest collects it last: a run that stops at its
first failure has then already run every other test.
"""
import numpy as np
import pytest

from block_quantized_matmul_gguf_gb300 import synth
from helpers import ABS, GEMM_REL, assert_within, bf16_tensor, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gguf_gb300 import build, qmm as q
    build.build_library()
    q.load()
    return q


def _with_workspace(qmm, wd, xd, m, n, k):
    ws = torch.empty(qmm.qmm_gemm_workspace_bytes(n, k), dtype=torch.uint8, device="cuda")
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    qmm.qmm_gemm_q4_0_ws(wd, xd, y, m, n, k, ws, ws.numel())
    torch.cuda.synchronize()
    return y


def test_prefill_without_workspace_two_calls_in_a_row(qmm, oracle_mod):
    # (m, n, k): one chunk at K = 2048, then K = 131072 (the largest the
    # scratch takes: 256 weight rows per chunk), N = 600 in chunks of 256,
    # 256 and 88 rows, over what the first call left in the scratch; both in
    # two phases (1100 tokens: five token blocks)
    calls = [(700, 1000, 2048, 11), (1100, 600, 131072, 12)]
    for i, (m, n, k, seed) in enumerate(calls):
        w, xb = synth.gemm_case(m, n, k, seed=seed)
        wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
        y_ws = _with_workspace(qmm, wd, xd, m, n, k)
        y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        qmm.qmm_gemm_q4_0_prefill(wd, xd, y, m, n, k)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert qmm.qmm_get_device_error() == 0
        if i > 0:  # warmed up: the call itself takes no device memory
            assert free_before - free_after < (1 << 20), (free_before, free_after)
        # the oracle on every output of the first call, on a sample of the
        # second (every chunk's first and last rows included)
        rng = np.random.default_rng(i)
        if i == 0:
            mi, ni = np.divmod(np.arange(m * n), n)
        else:
            mi = np.concatenate([rng.integers(0, m, 3000), [0, m - 1, 5, 9, m - 1]])
            ni = np.concatenate([rng.integers(0, n, 3000), [0, 255, 256, 511, 599]])
        y_ref, bound = oracle_mod.gemm_q4_0_at(w, xb, m, n, k, mi, ni)
        y_np, y_ws_np = y.cpu().numpy()[mi, ni], y_ws.cpu().numpy()[mi, ni]
        # against the workspace entry point, in the GEMM tolerance ...
        lim = GEMM_REL * bound + ABS
        diff = np.abs(y_np.astype(np.float64) - y_ws_np)
        assert np.all(diff <= lim), f"call {i}: {int((diff > lim).sum())} outputs off"
        # ... where both run the same kernels on the same weights: equal bits
        assert torch.equal(y, y_ws), f"call {i}: differs from qmm_gemm_q4_0_ws"
        assert_within(y_np, y_ref, bound, GEMM_REL, f"call {i} {m}x{n}x{k}")
