"""GPU parity: prefill GeGLU on the tensor cores, h = bf16(gelu_tanh(X.Wg^T) *
(X.Wu^T)), against the CPU oracle through the C ABI (qmm_gemm_q4_0_geglu)."""
import numpy as np
import pytest

from block_quantized_matmul_gguf_gb300 import synth
from helpers import GEMM_REL, assert_geglu_within, bf16_tensor, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BF16_OUT = 2.0 ** -8  # rounding of the stored h (bf16, nearest even), with margin


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gguf_gb300 import build, qmm as q
    build.build_library()
    q.load()
    return q


def _bf16_to_f32(bits):
    """bf16 bit patterns -> float32 (exact: the top half of a binary32)."""
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def _case(m, n, k, seed):
    wg = synth.q4_0_weights(n, k, seed=seed, stream=0)
    wu = synth.q4_0_weights(n, k, seed=seed, stream=1)
    xb = synth.activations_bf16(m, k, seed=seed, stream=2)
    return wg, wu, xb


def _run(qmm, wg, wu, xb, n, k):
    h = qmm.gemm_geglu_q4_0(to_dev(wg, torch), to_dev(wu, torch), bf16_tensor(xb, torch), n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    return _bf16_to_f32(h.cpu().numpy())


@pytest.mark.parametrize("m,n,k", [
    (1, 1, 256), (1, 64, 256), (300, 200, 512), (257, 130, 1024), (128, 128, 256),
    (512, 384, 2048), (700, 1000, 256), (33, 520, 768),
])
def test_gemm_geglu_matches_oracle(qmm, oracle_mod, m, n, k):
    # several pair tiles (128 features x 256 tokens), ragged token and
    # feature tails, several K stages
    wg, wu, xb = _case(m, n, k, m * 7 + n)
    h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, _bf16_to_f32(xb), m, n, k)
    assert_geglu_within(_run(qmm, wg, wu, xb, n, k), h_ref, g, u, bg, bu, f"{m}x{n}x{k}",
                        rel=GEMM_REL, out_rel=BF16_OUT)


def test_gemm_geglu_prefill_ffn_full_size_sampled(qmm, oracle_mod):
    """2048 prompt tokens through the 8192 x 2048 gate/up pair, sampled."""
    gate = next(p for p in synth.DECODE_LAYER if p.name == "gate")
    m, n, k = 2048, gate.n, gate.k
    wg, wu, xb = _case(m, n, k, 123)
    h = _run(qmm, wg, wu, xb, n, k)
    x = _bf16_to_f32(xb)
    rng = np.random.default_rng(9)
    mi = rng.integers(0, m, 4000)
    ni = rng.integers(0, n, 4000)
    h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0_at(wg, wu, x, m, n, k, mi, ni)
    assert_geglu_within(h[mi, ni], h_ref, g, u, bg, bu, "prefill ffn", rel=GEMM_REL,
                        out_rel=BF16_OUT)
    assert np.all(np.isfinite(h))


def test_gemm_geglu_agrees_with_the_plain_gemm(qmm):
    """g and u of the fused kernel are the plain GEMM's sums (same operands,
    same MMA sequence): h from the library's own two GEMM outputs agrees to
    the bf16 rounding of h."""
    m, n, k = 384, 512, 1024
    wg, wu, xb = (to_dev(a, torch) if a.dtype == np.uint8 else bf16_tensor(a, torch)
                  for a in _case(m, n, k, 5))
    h = qmm.gemm_geglu_q4_0(wg, wu, xb, n, k).view(torch.bfloat16).double()
    g = qmm.gemm_q4_0(wg, xb, n, k).double()
    u = qmm.gemm_q4_0(wu, xb, n, k).double()
    want = torch.nn.functional.gelu(g, approximate="tanh") * u
    err = (h - want).abs()
    assert bool((err <= 2.0 ** -8 * want.abs() + 1e-5 * (1 + g * g) * want.abs() + 1e-6).all())


def test_gemm_geglu_zero_gate_and_determinism(qmm):
    m, n, k = 300, 256, 512
    wz = np.zeros((n, k // 32, 18), np.uint8)
    wz[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    wz[:, :, 2:] = 0x88  # every gate weight zero -> g == 0 -> h == 0
    _, wu, xb = _case(m, n, k, 6)
    x = bf16_tensor(xb, torch)
    h = qmm.gemm_geglu_q4_0(to_dev(wz, torch), to_dev(wu, torch), x, n, k)
    # gelu(0) * u is a zero whose sign follows u: compare values, not bits
    assert torch.count_nonzero(h.view(torch.bfloat16)).item() == 0
    wg = to_dev(synth.q4_0_weights(n, k, seed=7), torch)
    wud = to_dev(wu, torch)
    a = qmm.gemm_geglu_q4_0(wg, wud, x, n, k)
    b = qmm.gemm_geglu_q4_0(wg, wud, x, n, k)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gemm_geglu_argument_checks(qmm):
    m, n, k = 4, 64, 256
    w = torch.zeros(n * (k // 32) * 18 + 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((m, k), dtype=torch.int16, device="cuda")
    h = torch.empty((m, n), dtype=torch.int16, device="cuda")
    for args, status in [((0, w, x, h, m, n, k), qmm.QMM_ERR_NULL),
                         ((w, w, x, 0, m, n, k), qmm.QMM_ERR_NULL),
                         ((w, w, x, h, 0, n, k), qmm.QMM_ERR_SHAPE),
                         ((w, w, x, h, m, n, 100), qmm.QMM_ERR_SHAPE),
                         ((w, w, x, h, m, n, 96), qmm.QMM_ERR_UNSUPPORTED),
                         ((w, w, x, h, m, n, 288), qmm.QMM_ERR_UNSUPPORTED),
                         ((w[1:].data_ptr(), w, x, h, m, n, k), qmm.QMM_ERR_ALIGN),
                         ((w, w, x, x, m, n, k), qmm.QMM_ERR_UNSUPPORTED)]:
        with pytest.raises(qmm.QmmError) as e:
            qmm.qmm_gemm_q4_0_geglu(*args)
        assert e.value.status == status, args
