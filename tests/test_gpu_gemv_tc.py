"""GPU parity of the tensor-core batched GEMV (qmm_gemv_q4_0_tc) against the
CPU oracle, in the fp32 GEMV's bound (1e-4 * sum|w*x| + 1e-6), plus exact
checks of its K order, its hi/lo split of x and its block scales."""
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


def _run(qmm, w, x, n, k):
    y = qmm.gemv_tc_q4_0(to_dev(w, torch), to_dev(x, torch), n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("m", list(range(1, 17)))
def test_gemv_tc_every_m(qmm, oracle_mod, m):
    # ragged rows (two 128-row tiles, the second partial), five K stages (no
    # cluster split)
    case = synth.gemv_case("q4_0", m, 203, 1280, seed=200 + m)
    y_ref, bound = oracle_mod.gemv_q4_0(case.w, case.x, m, case.n, case.k)
    assert_within(_run(qmm, case.w, case.x, case.n, case.k), y_ref, bound, GEMV_REL, f"tc m={m}")


@pytest.mark.parametrize("m,n,k", [
    (5, 300, 2048),     # 3 tiles, K split over a cluster of 8
    (8, 1000, 4096),    # cluster split with several tiles per cluster round
    (16, 129, 14336),   # the largest K at m > 8 (K split 8 ways)
    (3, 64, 36864),     # the largest K at m <= 8
    (9, 200, 2560),     # the largest K with no split at m > 8 (10 stages)
    (12, 20000, 2048),  # 157 tiles: more than one tile per cluster
    (1, 1, 256),        # one row, one stage
    (16, 4096, 256),    # one stage per row, many tiles
])
def test_gemv_tc_shapes(qmm, oracle_mod, m, n, k):
    case = synth.gemv_case("q4_0", m, n, k, seed=n + k + m)
    y_ref, bound = oracle_mod.gemv_q4_0(case.w, case.x, m, n, k)
    assert_within(_run(qmm, case.w, case.x, n, k), y_ref, bound, GEMV_REL, f"tc {m}x{n}x{k}")


@pytest.mark.parametrize("m", synth.BATCHED_M)
def test_gemv_tc_batched_decode_full(qmm, oracle_mod, m):
    """The batched decode workloads (8192 x 2048 and 2048 x 8192): every output."""
    for i, proj in enumerate(synth.BATCHED_SHAPES):
        case = synth.gemv_case("q4_0", m, proj.n, proj.k, seed=0, stream=30 + i)
        y_ref, bound = oracle_mod.gemv_q4_0(case.w, case.x, m, proj.n, proj.k)
        assert_within(_run(qmm, case.w, case.x, proj.n, proj.k), y_ref, bound, GEMV_REL,
                      f"tc {proj.name} m={m}")


def test_gemv_tc_one_hot_is_exact(qmm):
    """x row t = s_t * e_{c_t}: each y equals the dequantized weight times s_t
    with one fp32 rounding.  s = 1 checks the K order of both operands (the
    permuted slots of a block must pair each weight with its own activation);
    s = 1 + 2^-10 puts part of x in the low bf16 half (x_hi = 1, x_lo = 2^-10),
    which must be added back exactly."""
    n, k = 260, 1024
    case = synth.gemv_case("q4_0", 1, n, k, seed=7)
    w = to_dev(case.w, torch)
    deq = qmm.dequant("q4_0", w, n, k)
    cols = [0, 1, 2, 3, 4, 15, 16, 17, 18, 19, 31, 32, 255, 256, 511, 1023]
    for s in (1.0, 1.0 + 2.0 ** -10, -3.0):
        x = torch.zeros((len(cols), k), device="cuda")
        for t, c in enumerate(cols):
            x[t, c] = s
        y = qmm.gemv_tc_q4_0(w, x, n, k)
        torch.cuda.synchronize()
        want = deq[:, torch.tensor(cols, device="cuda")].t() * torch.tensor(s, device="cuda")
        assert torch.equal(y, want), s


def test_gemv_tc_deterministic_and_zero(qmm):
    case = synth.gemv_case("q4_0", 7, 2048, 2048, seed=5)
    w, x = to_dev(case.w, torch), to_dev(case.x, torch)
    a = qmm.gemv_tc_q4_0(w, x, 2048, 2048)
    b = qmm.gemv_tc_q4_0(w, x, 2048, 2048)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    z = qmm.gemv_tc_q4_0(w, torch.zeros_like(x), 2048, 2048)
    torch.cuda.synchronize()
    assert torch.count_nonzero(z).item() == 0


def test_gemv_tc_argument_checks(qmm):
    n, k = 64, 256
    w = torch.zeros(n * (k // 32) * 18 + 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((16, 37888), device="cuda")
    y = torch.empty((16, n), device="cuda")
    for args, status in [((0, x, y, 1, n, k), qmm.QMM_ERR_NULL),
                         ((w, x, y, 0, n, k), qmm.QMM_ERR_SHAPE),
                         ((w, x, y, 17, n, k), qmm.QMM_ERR_SHAPE),
                         ((w, x, y, 1, n, 288), qmm.QMM_ERR_UNSUPPORTED),      # k % 256
                         # a CTA's share of the activations would not fit shared memory
                         ((w, x, y, 9, n, 16384), qmm.QMM_ERR_UNSUPPORTED),
                         ((w, x, y, 16, n, 2816), qmm.QMM_ERR_UNSUPPORTED),   # 11 stages, no split
                         ((w, x, y, 8, n, 37888), qmm.QMM_ERR_UNSUPPORTED),
                         ((w[1:].data_ptr(), x, y, 1, n, k), qmm.QMM_ERR_ALIGN),
                         ((w, x.view(-1)[1:].data_ptr(), y, 1, n, k), qmm.QMM_ERR_ALIGN),
                         ((w, x, x, 1, n, k), qmm.QMM_ERR_UNSUPPORTED)]:   # y over x
        with pytest.raises(qmm.QmmError) as e:
            qmm.qmm_gemv_q4_0_tc(*args)
        assert e.value.status == status, args
