"""GPU tests of qmm_copy, the stream-ordered copy by the SMs that moves a
decode step's activations in from page-locked host memory and its outputs
back: every byte at every size and alignment in each direction, the ordering
against the GEMV launches around it (with programmatic dependent launch),
the same inside a captured CUDA graph, and the refusal of pageable memory."""
import numpy as np
import pytest

from block_quantized_matmul_gguf_gb300 import synth
from helpers import GEMV_REL, assert_within, to_dev

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


def _bytes(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8))


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 4099, (1 << 20) + 5])
@pytest.mark.parametrize("offsets", [(0, 0), (1, 3), (16, 32)])
def test_copy_every_byte(qmm, direction, nbytes, offsets):
    so, do = offsets
    pad = 64
    src_h = _bytes(nbytes + pad, nbytes).pin_memory()
    src = src_h if direction == "h2d" else src_h.cuda()
    dst_fill = 0xA5
    dst = torch.full((nbytes + pad,), dst_fill, dtype=torch.uint8)
    dst = dst.pin_memory() if direction == "d2h" else dst.cuda()
    qmm.qmm_copy(dst.data_ptr() + do, src.data_ptr() + so, nbytes)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    got = dst.cpu()
    want = src_h[so:so + nbytes]
    assert torch.equal(got[do:do + nbytes], want)
    # nothing written outside the range
    assert (got[:do] == dst_fill).all() and (got[do + nbytes:] == dst_fill).all()


def test_copy_refuses_pageable_host_memory(qmm):
    host = torch.zeros(256, dtype=torch.uint8)  # not pinned
    dev = torch.ones(256, dtype=torch.uint8, device="cuda")
    L = qmm.load()
    assert L.qmm_copy(host.data_ptr(), dev.data_ptr(), 256, None) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_copy(dev.data_ptr(), host.data_ptr(), 256, None) == qmm.QMM_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        qmm.qmm_copy(dev, host, 256)
    torch.cuda.synchronize()
    assert (host == 0).all()


def _step(qmm, w, x_dev, y_dev, x_host, y_host, n, k, m, stream):
    """Activations in, one GEMV, outputs out: three launches in stream order."""
    qmm.qmm_copy(x_dev, x_host, x_host.numel() * 4, stream)
    qmm.qmm_gemv_q4_0(w, x_dev, y_dev, m, n, k, stream)
    qmm.qmm_copy(y_host, y_dev, y_host.numel() * 4, stream)


@pytest.mark.parametrize("graph", [False, True])
def test_copy_orders_with_the_gemv_launches(qmm, oracle_mod, graph):
    """Each round puts new activations in the same device buffer and reads
    the GEMV's output back: the copy-in must not overtake the previous GEMV's
    reads, and the copy-out must see this GEMV's writes.  Run eagerly and as
    a replayed CUDA graph; every round against the oracle."""
    m, n, k = 2, 2048, 2048
    w = synth.q4_0_weights(n, k, seed=31)
    wd = to_dev(w, torch)
    xs = [synth.activations_f32(m, k, seed=31, stream=s) for s in range(4)]
    x_host = torch.empty((m, k), dtype=torch.float32).pin_memory()
    y_host = torch.empty((m, n), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((m, k), dtype=torch.float32, device="cuda")
    y_dev = torch.empty((m, n), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = None
    if graph:
        x_host.copy_(torch.from_numpy(xs[0]))
        with torch.cuda.stream(stream):
            _step(qmm, wd, x_dev, y_dev, x_host, y_host, n, k, m, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            _step(qmm, wd, x_dev, y_dev, x_host, y_host, n, k, m, stream)
        torch.cuda.synchronize()
    for r, x in enumerate(xs):
        x_host.copy_(torch.from_numpy(x))
        y_host.fill_(float("nan"))
        if graph:
            g.replay()
        else:
            with torch.cuda.stream(stream):
                _step(qmm, wd, x_dev, y_dev, x_host, y_host, n, k, m, stream)
        torch.cuda.synchronize()
        assert qmm.qmm_get_device_error() == 0
        y_ref, bound = oracle_mod.gemv_q4_0(w, x, m, n, k)
        assert_within(y_host.numpy(), y_ref, bound, GEMV_REL, f"round {r} graph={graph}")
