"""GPU parity of the tcgen05 prefill GEMM with Q8_0 weights (qmm_gemm_q8_0)
against the CPU oracle (2e-3 bound), plus exact checks of its decode and
bf16 rounding."""
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


def _bf16_to_f32(bits):
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def _gemm(qmm, w, xb, m, n, k):
    y = qmm.gemm("q8_0", to_dev(w, torch), bf16_tensor(xb, torch), n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    return y


def _every_byte_weights(n, k):
    """Q8_0 rows in which every byte value (q = -128..127) appears at every
    position class, with ordinary, tiny (subnormal), large and negative d."""
    nb = k // 32
    blocks = np.zeros((n, nb, 34), np.uint8)
    scales = [0x3C00, 0x0001, 0x03FF, 0x7BFF, 0xB800, 0x1234, 0x8001, 0x2E66]
    for r in range(n):
        for b in range(nb):
            d = scales[(r + b) % len(scales)]
            blocks[r, b, 0], blocks[r, b, 1] = d & 0xFF, d >> 8
            blocks[r, b, 2:] = (np.arange(32) * 8 + r * 5 + b * 3) % 256
    return blocks.reshape(n, -1)


def test_gemm_q8_0_one_hot_gives_every_weight_bf16_rounded(qmm):
    """X = I (k x k): Y[i][n] = bf16(w[n][i]) exactly for every weight of W,
    against torch's RNE of the bit-exact dequantisation."""
    m = n = k = 256
    w = _every_byte_weights(n, k)
    wd = to_dev(w, torch)
    deq = qmm.dequant("q8_0", wd, n, k)
    x = np.zeros((m, k), dtype=np.uint16)
    x[np.arange(m), np.arange(m)] = 0x3F80  # bf16 1.0
    y = _gemm(qmm, w, x, m, n, k)
    want = deq.to(torch.bfloat16).float().t()
    assert torch.equal(y, want)


@pytest.mark.parametrize("m,n,k", [
    (128, 256, 256), (1, 256, 256), (129, 260, 512), (300, 1000, 768), (256, 512, 2048),
    (77, 4, 256), (513, 768, 1024),
])
def test_gemm_q8_0_parity_small(qmm, oracle_mod, m, n, k):
    w = synth.q8_0_weights(n, k, seed=m + n, stream=0)
    xb = synth.activations_bf16(m, k, seed=m + n, stream=1)
    y = _gemm(qmm, w, xb, m, n, k).cpu().numpy()
    y_ref, bound = oracle_mod.gemv_q8_0(w, _bf16_to_f32(xb), m, n, k)
    assert_within(y, y_ref, bound, GEMM_REL, f"q8_0 gemm {m}x{n}x{k}")


def test_gemm_q8_0_lm_head_prompt_sampled(qmm, oracle_mod):
    """512 prompt positions through the 262144 x 2048 Q8_0 LM head, sampled."""
    p = synth.LM_HEAD
    m = 512
    w = synth.q8_0_weights(p.n, p.k, seed=0, stream=50)
    xb = synth.activations_bf16(m, p.k, seed=3, stream=1)
    y = _gemm(qmm, w, xb, m, p.n, p.k)
    rng = np.random.default_rng(11)
    mi = np.concatenate([rng.integers(0, m, 3000), [0, m - 1]])
    ni = np.concatenate([rng.integers(0, p.n, 3000), [p.n - 1, 0]])
    got = y[torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()].cpu().numpy()
    y_ref, bound = oracle_mod.gemv_q8_0_at(w, _bf16_to_f32(xb), m, p.n, p.k, mi, ni)
    assert_within(got, y_ref, bound, GEMM_REL, "q8_0 lm head prompt")
    assert bool(torch.isfinite(y).all())


def test_gemm_q8_0_deterministic_and_zeros(qmm):
    m, n, k = 384, 512, 1024
    w = synth.q8_0_weights(n, k, seed=4)
    xb = synth.activations_bf16(m, k, seed=4, stream=1)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    a = qmm.gemm("q8_0", wd, xd, n, k)
    b = qmm.gemm("q8_0", wd, xd, n, k)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    wz = np.zeros((n, k // 32, 34), np.uint8)
    wz[:, :, 0:2] = np.frombuffer(np.float16(0.01).tobytes(), np.uint8)  # q = 0
    y = _gemm(qmm, wz.reshape(n, -1), xb, m, n, k)
    assert torch.count_nonzero(y).item() == 0


def test_gemm_q8_0_argument_checks(qmm):
    m, n, k = 4, 64, 256
    w = torch.zeros(n * (k // 32) * 34 + 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((m, k), dtype=torch.int16, device="cuda")
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    for args, status in [((0, x, y, m, n, k), qmm.QMM_ERR_NULL),
                         ((w, x, y, m, n, 100), qmm.QMM_ERR_SHAPE),
                         ((w, x, y, m, n, 96), qmm.QMM_ERR_UNSUPPORTED),
                         ((w, x, x, m, n, k), qmm.QMM_ERR_UNSUPPORTED),   # y over x
                         ((w[1:].data_ptr(), x, y, m, n, k), qmm.QMM_ERR_ALIGN)]:
        with pytest.raises(qmm.QmmError) as e:
            qmm.qmm_gemm_q8_0(*args)
        assert e.value.status == status, args
