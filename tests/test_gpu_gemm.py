"""GPU parity of the tcgen05 prefill GEMM against the CPU oracle (2e-3 bound),
plus exact checks of its bf16 weight rounding and operand layout."""
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


# The bf16 rounding of each weight is the GEMM's error budget.  Its worst
# case (2^-9 relative per weight, all of one sign) would fill the 2e-3 bound;
# the expected error is far smaller.  Each full-size product records the
# largest fraction of the tolerance it uses, max |err| / (2e-3 * sum|w*x| +
# 1e-6), and must stay at or below a quarter of it (else the tiles would have
# to move to fp16, whose rounding is 2^-12).
C9_MAX_FRACTION = 0.25


def tolerance_fraction(y, y_ref, bound, rel=GEMM_REL):
    err = np.abs(np.asarray(y, np.float64) - y_ref)
    return float(np.max(err / (rel * bound + ABS))), float(np.max(err / np.maximum(bound, 1e-300)))


@pytest.mark.parametrize("shape", synth.PREFILL_SHAPES, ids=lambda p: f"{p.n}x{p.k}")
def test_gemm_full_size_full_output(qmm, oracle_mod, shape):
    """2048-token prefill at both weight shapes: every output against the
    oracle, plus the fraction of the tolerance used."""
    m = synth.PREFILL_M
    w, xb = synth.gemm_case(m, shape.n, shape.k, seed=0, stream=70 + synth.PREFILL_SHAPES.index(shape))
    y = _gemm(qmm, w, xb, m, shape.n, shape.k).cpu().numpy()
    y_ref, bound = oracle_mod.gemm_q4_0(w, xb, m, shape.n, shape.k)
    assert_within(y, y_ref, bound, GEMM_REL, f"gemm {m}x{shape.n}x{shape.k}")
    frac, rel = tolerance_fraction(y, y_ref, bound)
    print(f"C9 gemm {m}x{shape.n}x{shape.k}: max |err|/(2e-3 bound + 1e-6) = {frac:.4g}, "
          f"max |err|/bound = {rel:.4g}")
    assert frac <= C9_MAX_FRACTION, frac


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


def _bf16_to_f32(bits):
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n", [1, 3, 5, 1001])
@pytest.mark.parametrize("path", ["q4_0", "q8_0", "q4_0_ws", "q8_0_ws", "q4_0_prefill"])
def test_gemm_any_n(qmm, oracle_mod, path, n):
    """Any n >= 1: ragged weight tiles and outputs whose rows are not 16-byte
    multiples, on the fused (m = 300), two-phase (m = 520) and static-scratch
    paths, with y one float past an allocation's start (4-byte aligned)."""
    fmt = path[:4]
    m = 520 if ("ws" in path or "prefill" in path) else 300
    k = 512
    w = (synth.q4_0_weights if fmt == "q4_0" else synth.q8_0_weights)(n, k, seed=n, stream=1)
    xb = synth.activations_bf16(m, k, seed=n, stream=2)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    buf = torch.full((m * n + 1,), float("nan"), dtype=torch.float32, device="cuda")
    y = buf[1:]
    f = getattr(qmm, "qmm_gemm_" + path.replace("_ws", ""))
    if path.endswith("_ws"):
        ws = torch.empty(qmm.qmm_gemm_workspace_bytes(n, k), dtype=torch.uint8, device="cuda")
        getattr(qmm, f"qmm_gemm_{fmt}_ws")(wd, xd, y.data_ptr(), m, n, k, ws, ws.numel())
    else:
        f(wd, xd, y.data_ptr(), m, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.isnan(buf[:1]).all()  # nothing written before y
    if fmt == "q4_0":
        y_ref, bound = oracle_mod.gemm_q4_0(w, xb, m, n, k)
    else:
        y_ref, bound = oracle_mod.gemv_q8_0(w, _bf16_to_f32(xb), m, n, k)
    assert_within(y.view(m, n).cpu().numpy(), y_ref, bound, GEMM_REL, f"{path} n={n}")
