"""GPU parity of the tcgen05 prefill GEMM against the CPU oracle (2e-3 bound),
plus exact checks of its bf16 weight rounding and operand layout."""
import numpy as np
import pytest

from block_quantized_matmul_gguf_gb300 import synth
from helpers import GEMM_REL, assert_within, bf16_tensor, to_dev

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


def _gemm(qmm, w, xb, m, n, k):
    y = qmm.gemm_q4_0(to_dev(w, torch), bf16_tensor(xb, torch), n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    return y


def test_gemm_one_hot_rows_give_bf16_rounded_weights(qmm):
    """X row i = e_{c_i}: Y[i][n] = bf16(w[n][c_i]) exactly (one nonzero
    product, fp32 sum).  Pins the bf16 rounding (against torch's RNE of the
    bit-exact dequantisation) and the K / N placement in both operands."""
    m, n, k = 128, 512, 512
    w, _ = synth.gemm_case(1, n, k, seed=31)
    wd = to_dev(w, torch)
    deq = qmm.dequant("q4_0", wd, n, k)
    cols = (np.arange(m) * 37 + 5) % k
    x = np.zeros((m, k), dtype=np.uint16)
    x[np.arange(m), cols] = 0x3F80  # bf16 1.0
    y = _gemm(qmm, w, x, m, n, k)
    want = deq.to(torch.bfloat16).float()[:, torch.from_numpy(cols).cuda()].t()
    assert torch.equal(y, want)


def test_gemm_scaled_one_hot(qmm):
    """X row i = 2^j e_c (power of two, exact) for several rows per column."""
    m, n, k = 256, 256, 256
    w, _ = synth.gemm_case(1, n, k, seed=32)
    wd = to_dev(w, torch)
    deq = qmm.dequant("q4_0", wd, n, k).to(torch.bfloat16).float()
    cols = (np.arange(m) * 11) % k
    scale = 2.0 ** ((np.arange(m) % 7) - 3)
    x = np.zeros((m, k), dtype=np.float32)
    x[np.arange(m), cols] = scale
    xb = synth.f32_to_bf16_bits(x)
    y = _gemm(qmm, w, xb, m, n, k)
    want = deq[:, torch.from_numpy(cols).cuda()].t() * torch.from_numpy(scale).float().cuda()[:, None]
    assert torch.equal(y, want)


@pytest.mark.parametrize("m,n,k", [
    (128, 256, 256), (1, 256, 256), (129, 260, 512), (300, 1000, 768), (256, 512, 2048),
    (77, 4, 256), (513, 768, 1024),
])
def test_gemm_parity_small(qmm, oracle_mod, m, n, k):
    w, xb = synth.gemm_case(m, n, k, seed=m + n + k)
    y = _gemm(qmm, w, xb, m, n, k).cpu().numpy()
    y_ref, bound = oracle_mod.gemm_q4_0(w, xb, m, n, k)
    r = assert_within(y, y_ref, bound, GEMM_REL, f"gemm {m}x{n}x{k}")
    print(f"gemm {m}x{n}x{k}: max |err|/bound = {r:.3g}")


@pytest.mark.parametrize("shape", synth.PREFILL_SHAPES, ids=lambda p: f"{p.n}x{p.k}")
def test_gemm_full_size_sampled(qmm, oracle_mod, shape):
    m = synth.PREFILL_M
    w, xb = synth.gemm_case(m, shape.n, shape.k, seed=0, stream=70 + synth.PREFILL_SHAPES.index(shape))
    y = _gemm(qmm, w, xb, m, shape.n, shape.k).cpu().numpy()
    rng = np.random.default_rng(5)
    mi = np.concatenate([rng.integers(0, m, 1500), [0, m - 1, m - 1, 0]])
    ni = np.concatenate([rng.integers(0, shape.n, 1500), [0, shape.n - 1, 0, shape.n - 1]])
    y_ref, bound = oracle_mod.gemm_q4_0_at(w, xb, m, shape.n, shape.k, mi, ni)
    r = assert_within(y[mi, ni], y_ref, bound, GEMM_REL, f"gemm {m}x{shape.n}x{shape.k}")
    print(f"full-size gemm {shape.n}x{shape.k}: max |err|/bound = {r:.3g}")
    assert np.all(np.isfinite(y))


def test_gemm_deterministic(qmm):
    m, n, k = 384, 512, 1024
    w, xb = synth.gemm_case(m, n, k, seed=4)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    a = qmm.gemm_q4_0(wd, xd, n, k)
    b = qmm.gemm_q4_0(wd, xd, n, k)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gemm_zero_weights_and_zero_x(qmm):
    m, n, k = 200, 256, 512
    w = np.zeros((n, k // 32, 18), np.uint8)
    w[:, :, 0:2] = np.frombuffer(np.float16(0.01).tobytes(), np.uint8)
    w[:, :, 2:] = 0x88  # every nibble 8 -> weight 0
    xb = synth.activations_bf16(m, k, seed=1)
    y = _gemm(qmm, w, xb, m, n, k)
    assert torch.count_nonzero(y).item() == 0
    w2, _ = synth.gemm_case(1, n, k, seed=2)
    y = _gemm(qmm, w2, np.zeros((m, k), np.uint16), m, n, k)
    assert torch.count_nonzero(y).item() == 0
