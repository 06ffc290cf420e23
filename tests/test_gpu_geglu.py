"""GPU parity: fused GeGLU decode h = gelu_tanh(x.Wg^T) * (x.Wu^T) against
the CPU oracle, through the C ABI (qmm_gemv_q4_0_geglu)."""
import numpy as np
import pytest

from block_quantized_matmul_gguf_gb300 import synth
from helpers import assert_geglu_within, to_dev

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


def _case(m, n, k, seed):
    wg = synth.q4_0_weights(n, k, seed=seed, stream=0)
    wu = synth.q4_0_weights(n, k, seed=seed, stream=1)
    x = synth.activations_f32(m, k, seed=seed, stream=2)
    return wg, wu, x


def _run(qmm, wg, wu, x, n, k):
    return qmm.geglu_q4_0(to_dev(wg, torch), to_dev(wu, torch), to_dev(x, torch), n, k).cpu().numpy()


def _check(qmm, oracle_mod, m, n, k, seed, what):
    wg, wu, x = _case(m, n, k, seed)
    h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, x, m, n, k)
    assert_geglu_within(_run(qmm, wg, wu, x, n, k), h_ref, g, u, bg, bu, what)


@pytest.mark.parametrize("m", list(range(1, 17)))
def test_geglu_every_m(qmm, oracle_mod, m):
    # ragged N (not a multiple of 32 or 16), several K chunks
    _check(qmm, oracle_mod, m, 203, 1280, 300 + m, f"m={m}")


@pytest.mark.parametrize("m,n,k", [
    (1, 1, 256), (1, 37, 256), (3, 31, 512), (2, 64, 16384), (1, 257, 8192),
    (4, 1000, 2048), (5, 999, 768), (16, 64, 16384), (8, 300, 4096), (1, 4096, 2048),
])
def test_geglu_shapes(qmm, oracle_mod, m, n, k):
    # two lanes per row (small problems), one lane per row, cluster K splits
    # (small N, large K), ragged tails
    _check(qmm, oracle_mod, m, n, k, m * 31 + n, f"{m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(1, 40, 96), (3, 33, 32), (2, 70, 1312)])
def test_geglu_k_not_multiple_of_256_takes_bytewise(qmm, oracle_mod, m, n, k):
    _check(qmm, oracle_mod, m, n, k, n + k, f"bytewise {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(16, 40, 65536), (10, 70, 32768)])
def test_geglu_very_large_k_falls_back(qmm, oracle_mod, m, n, k):
    _check(qmm, oracle_mod, m, n, k, m + n, f"large-k {m}x{n}x{k}")


def test_geglu_unaligned_weights_and_x(qmm, oracle_mod):
    m, n, k = 2, 100, 512
    wg, wu, x = _case(m, n, k, 77)
    h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, x, m, n, k)
    bufg = torch.zeros(wg.size + 3, dtype=torch.uint8, device="cuda")
    bufg[3:] = to_dev(wg.reshape(-1), torch)
    bufx = torch.zeros(m * k + 1, dtype=torch.float32, device="cuda")
    bufx[1:] = to_dev(x.reshape(-1), torch)
    h = torch.empty((m, n), dtype=torch.float32, device="cuda")
    qmm.qmm_gemv_q4_0_geglu(bufg[3:].data_ptr(), to_dev(wu, torch), bufx[1:].data_ptr(), h, m, n, k)
    assert_geglu_within(h.cpu().numpy(), h_ref, g, u, bg, bu, "unaligned")


def test_geglu_decode_ffn_full_size_sampled(qmm, oracle_mod):
    """The decode layer's gate/up pair (8192 x 2048 each) at M = 1 and 8,
    checked on sampled outputs against the oracle's per-output products."""
    gate = next(p for p in synth.DECODE_LAYER if p.name == "gate")
    n, k = gate.n, gate.k
    wg = synth.q4_0_weights(n, k, seed=90, stream=0)
    wu = synth.q4_0_weights(n, k, seed=90, stream=1)
    rng = np.random.default_rng(5)
    for m in (1, 8):
        x = synth.activations_f32(m, k, seed=91 + m)
        h = _run(qmm, wg, wu, x, n, k)
        mi = rng.integers(0, m, 3000)
        ni = rng.integers(0, n, 3000)
        h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0_at(wg, wu, x, m, n, k, mi, ni)
        assert_geglu_within(h[mi, ni], h_ref, g, u, bg, bu, f"ffn m={m}")
        assert np.all(np.isfinite(h))


def test_geglu_zero_gate_gives_exact_zero_and_is_deterministic(qmm):
    n, k = 300, 2048
    wz = np.zeros((n, k // 32, 18), np.uint8)
    wz[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    wz[:, :, 2:] = 0x88  # every weight zero -> g == 0 -> h == 0
    wu = synth.q4_0_weights(n, k, seed=3)
    x = to_dev(synth.activations_f32(4, k, seed=4), torch)
    h = qmm.geglu_q4_0(to_dev(wz, torch), to_dev(wu, torch), x, n, k)
    assert torch.count_nonzero(h).item() == 0
    wg = to_dev(synth.q4_0_weights(n, k, seed=5), torch)
    wud = to_dev(wu, torch)
    a = qmm.geglu_q4_0(wg, wud, x, n, k)
    b = qmm.geglu_q4_0(wg, wud, x, n, k)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_geglu_matches_separate_gemvs(qmm):
    """The fused call reproduces gelu(gemv(gate)) * gemv(up) made of the
    library's own GEMV outputs up to the fp32 GELU (same sums, same order
    is not promised, so a relative tolerance)."""
    m, n, k = 2, 512, 2048
    wg, wu, x = (to_dev(a, torch) for a in _case(m, n, k, 8))
    h = qmm.geglu_q4_0(wg, wu, x, n, k)
    g = qmm.gemv("q4_0", wg, x, n, k).double()
    u = qmm.gemv("q4_0", wu, x, n, k).double()
    want = torch.nn.functional.gelu(g, approximate="tanh") * u
    torch.testing.assert_close(h.double(), want, rtol=1e-4, atol=1e-4)


def test_geglu_argument_checks(qmm):
    n, k = 64, 256
    w = torch.zeros(n * (k // 32) * 18, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, k), device="cuda")
    h = torch.empty((1, n), device="cuda")
    for args, status in [((0, w, x, h, 1, n, k), qmm.QMM_ERR_NULL),
                         ((w, 0, x, h, 1, n, k), qmm.QMM_ERR_NULL),
                         ((w, w, x, h, 17, n, k), qmm.QMM_ERR_SHAPE),
                         ((w, w, x, h, 1, n, 100), qmm.QMM_ERR_SHAPE),
                         ((w, w, x, x, 1, n, k), qmm.QMM_ERR_UNSUPPORTED)]:
        with pytest.raises(qmm.QmmError) as e:
            qmm.qmm_gemv_q4_0_geglu(*args)
        assert e.value.status == status
