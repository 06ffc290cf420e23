"""GPU parity of the two-phase prefill GEMM (weights dequantised once into a
bf16 workspace, then a shared-memory-operand tensor-core GEMM) against the
CPU oracle, and bit-for-bit against the fused kernel (same weights, same MMA
sequence)."""
import numpy as np
import pytest

from block_quantized_matmul_gguf_gb300 import synth
from helpers import GEMM_REL, assert_geglu_within, assert_within, bf16_tensor, to_dev

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


def _ws(qmm, n, k, geglu=False):
    return torch.empty(qmm.qmm_gemm_workspace_bytes(n, k, geglu), dtype=torch.uint8, device="cuda")


def _weights(fmt, n, k, seed, stream=0):
    return (synth.q4_0_weights if fmt == "q4_0" else synth.q8_0_weights)(n, k, seed=seed, stream=stream)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
# two phases from the third 256-token block on when the fused kernel would
# not split K (its partial products would not fit, or K is too short), and
# from the fifth block in any case
@pytest.mark.parametrize("m,n,k", [(520, 4, 256), (600, 260, 512), (513, 768, 1024),
                                   (700, 1000, 256), (1024, 384, 2048), (1100, 136, 4096)])
def test_two_phase_matches_oracle_and_fused(qmm, oracle_mod, fmt, m, n, k):
    w = _weights(fmt, n, k, seed=m + n)
    xb = synth.activations_bf16(m, k, seed=m + n, stream=5)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y2 = qmm.gemm(fmt, wd, xd, n, k, workspace=_ws(qmm, n, k))
    y1 = qmm.gemm(fmt, wd, xd, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    y_ref, bound = f(w, _bf16_to_f32(xb), m, n, k)
    assert_within(y2.cpu().numpy(), y_ref, bound, GEMM_REL, f"two-phase {fmt} {m}x{n}x{k}")
    assert torch.equal(y2, y1), "two-phase and fused results differ"


@pytest.mark.parametrize("shape", synth.PREFILL_SHAPES, ids=lambda p: f"{p.n}x{p.k}")
def test_two_phase_full_size_equals_fused(qmm, oracle_mod, shape):
    """The 2048-token prefill at both weight shapes, on the inputs whose every
    output the fused kernel's full-size test checks against the oracle: the
    workspace and static-scratch calls give the fused kernel's exact bits."""
    m = synth.PREFILL_M
    w, xb = synth.gemm_case(m, shape.n, shape.k, seed=0,
                            stream=70 + synth.PREFILL_SHAPES.index(shape))
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y2 = qmm.gemm("q4_0", wd, xd, shape.n, shape.k, workspace=_ws(qmm, shape.n, shape.k))
    y1 = qmm.gemm("q4_0", wd, xd, shape.n, shape.k)
    y3 = torch.empty_like(y1)
    qmm.qmm_gemm_q4_0_prefill(wd, xd, y3, m, shape.n, shape.k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(y2, y1) and torch.equal(y3, y1)
    rng = np.random.default_rng(3)
    mi = rng.integers(0, m, 2000)
    ni = rng.integers(0, shape.n, 2000)
    y_ref, bound = oracle_mod.gemm_q4_0_at(w, xb, m, shape.n, shape.k, mi, ni)
    assert_within(y2[torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()].cpu().numpy(),
                  y_ref, bound, GEMM_REL, "two-phase full size")


@pytest.mark.parametrize("m,n,k", [(600, 200, 512), (520, 384, 2048), (700, 1000, 256), (300, 72, 4096)])
def test_two_phase_geglu(qmm, oracle_mod, m, n, k):
    wg = synth.q4_0_weights(n, k, seed=m, stream=0)
    wu = synth.q4_0_weights(n, k, seed=m, stream=1)
    xb = synth.activations_bf16(m, k, seed=m, stream=2)
    a, b, xd = to_dev(wg, torch), to_dev(wu, torch), bf16_tensor(xb, torch)
    h2 = qmm.gemm_geglu_q4_0(a, b, xd, n, k, workspace=_ws(qmm, n, k, geglu=True))
    h1 = qmm.gemm_geglu_q4_0(a, b, xd, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(h2, h1), "two-phase and fused GeGLU differ"
    h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, _bf16_to_f32(xb), m, n, k)
    assert_geglu_within(_bf16_to_f32(h2.cpu().numpy()), h_ref, g, u, bg, bu, f"{m}x{n}x{k}",
                        rel=GEMM_REL, out_rel=2.0 ** -8)


@pytest.mark.parametrize("m,n,k", [(256, 512, 512), (512, 512, 2048), (256, 512, 4096)])
def test_short_prompt_with_a_workspace(qmm, oracle_mod, m, n, k):
    """Short prompts run the fused kernel; where its tiles leave the GPU idle
    they split K through the workspace (512 x 2048 at m = 512: 2 parts;
    512 x 4096 at m = 256: 4 parts; 512 x 512: two raw stages, too few to
    split).  Same bound as the unsplit product, identical to the
    static-scratch entry, deterministic."""
    w, xb = synth.gemm_case(m, n, k, seed=9)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    ws = _ws(qmm, n, k)
    ws.fill_(0xA5)
    y = qmm.gemm("q4_0", wd, xd, n, k, workspace=ws)
    y2 = qmm.gemm("q4_0", wd, xd, n, k, workspace=ws)
    y3 = _prefill(qmm, wd, xd, m, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(y, y2) and torch.equal(y, y3)
    y_ref, bound = oracle_mod.gemm_q4_0(w, xb, m, n, k)
    assert_within(y.cpu().numpy(), y_ref, bound, GEMM_REL, f"short {m}x{n}x{k}")


@pytest.mark.parametrize("fmt,m,n,k", [("q4_0", 256, 2048, 8192), ("q4_0", 256, 8192, 2048),
                                       ("q4_0", 77, 1000, 4096), ("q8_0", 200, 1024, 2048),
                                       ("q4_0", 1, 4096, 2048), ("q4_0", 128, 300, 1280)])
def test_short_prompt_k_split(qmm, oracle_mod, fmt, m, n, k):
    """K split for short prompts (8 parts at 256 x 2048 x 8192, 2 at
    256 x 8192 x 2048, 4 with ragged tokens and rows, 2 for Q8_0, 2 at one
    token; 1280 has five raw stages, so no split): every output against the
    oracle, and against the unsplit fused product within the same bound."""
    w = _weights(fmt, n, k, seed=m + n)
    xb = synth.activations_bf16(m, k, seed=m + n, stream=6)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y = qmm.gemm(fmt, wd, xd, n, k, workspace=_ws(qmm, n, k))
    y1 = qmm.gemm(fmt, wd, xd, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    y_ref, bound = f(w, _bf16_to_f32(xb), m, n, k)
    assert_within(y.cpu().numpy(), y_ref, bound, GEMM_REL, f"split {fmt} {m}x{n}x{k}")
    assert_within(y1.cpu().numpy(), y_ref, bound, GEMM_REL, f"fused {fmt} {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k,form", [(1024, 2048, 8192, "split"), (600, 2048, 8192, "split"),
                                        (768, 4096, 4096, "two"), (384, 8192, 8192, "fused")])
def test_medium_prompt_form(qmm, oracle_mod, m, n, k, form):
    """Two to four token blocks: at 2048 x 8192 the fused kernel's 24-32 pair
    tiles split K in two (one phase, the workspace holds the parts); at
    4096 x 4096 with three blocks (48 tiles) no split fits one round and the
    product runs in two phases; 8192 x 8192 with two blocks runs the fused
    kernel unsplit.  The last two give the workspace-free fused call's bits.
    Sampled outputs against the oracle; the static-scratch entry gives the
    same bits as the workspace entry in every form."""
    w, xb = synth.gemm_case(m, n, k, seed=m + 3)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y = qmm.gemm("q4_0", wd, xd, n, k, workspace=_ws(qmm, n, k))
    y3 = _prefill(qmm, wd, xd, m, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(y, y3)
    if form != "split":
        assert torch.equal(y, qmm.gemm("q4_0", wd, xd, n, k))
    rng = np.random.default_rng(m)
    mi = np.concatenate([rng.integers(0, m, 1500), [0, m - 1, m - 1]])
    ni = np.concatenate([rng.integers(0, n, 1500), [n - 1, 0, n - 1]])
    y_ref, bound = oracle_mod.gemm_q4_0_at(w, xb, m, n, k, mi, ni)
    assert_within(y.cpu().numpy()[mi, ni], y_ref, bound, GEMM_REL, f"{form} {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k,form", [(1024, 2048, 8192, "split"), (768, 4096, 4096, "two")])
def test_medium_prompt_form_q8_0(qmm, oracle_mod, m, n, k, form):
    """The same choice of form for Q8_0 weights: at 2048 x 8192 the fused kernel
    splits K through the workspace, at 4096 x 4096 with three token blocks the
    product runs in two phases with the fused kernel's bits.  Sampled outputs
    against the oracle."""
    w = _weights("q8_0", n, k, seed=m + 7)
    xb = synth.activations_bf16(m, k, seed=m + 7, stream=5)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y = qmm.gemm("q8_0", wd, xd, n, k, workspace=_ws(qmm, n, k))
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    if form == "two":
        assert torch.equal(y, qmm.gemm("q8_0", wd, xd, n, k))
    rng = np.random.default_rng(m + 1)
    mi = np.concatenate([rng.integers(0, m, 1500), [0, m - 1]])
    ni = np.concatenate([rng.integers(0, n, 1500), [n - 1, 0]])
    y_ref, bound = oracle_mod.gemv_q8_0_at(w, _bf16_to_f32(xb), m, n, k, mi, ni)
    assert_within(y.cpu().numpy()[mi, ni], y_ref, bound, GEMM_REL, f"q8_0 {form} {m}x{n}x{k}")


def test_workspace_argument_checks(qmm):
    m, n, k = 600, 64, 256
    w = torch.zeros(n * (k // 32) * 18, dtype=torch.uint8, device="cuda")
    x = torch.zeros((m, k), dtype=torch.int16, device="cuda")
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    need = qmm.qmm_gemm_workspace_bytes(n, k)  # 32 KB: y (153.6 KB) covers it
    assert need == n * k * 2
    assert qmm.qmm_gemm_workspace_bytes(n, k, geglu=True) == (n + 63) // 64 * 128 * k * 2
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    for args, status in [((w, x, y, m, n, k, ws, need - 1), qmm.QMM_ERR_SHAPE),
                         ((w, x, y, m, n, k, ws[8:].data_ptr(), need), qmm.QMM_ERR_ALIGN),
                         ((w, x, y, m, n, k, y, need), qmm.QMM_ERR_UNSUPPORTED)]:
        with pytest.raises(qmm.QmmError) as e:
            qmm.qmm_gemm_q4_0_ws(*args)
        assert e.value.status == status, args


# ---- the same product on the library's own scratch (no workspace argument) ----

def _prefill(qmm, w, x, m, n, k):
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    qmm.qmm_gemm_q4_0_prefill(w, x, y, m, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    return y


@pytest.mark.parametrize("m,n,k", [(600, 260, 512), (1024, 384, 2048), (200, 512, 512), (1100, 256, 4096)])
def test_prefill_static_scratch_equals_fused(qmm, oracle_mod, m, n, k):
    w, xb = synth.gemm_case(m, n, k, seed=m + 1)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y = _prefill(qmm, wd, xd, m, n, k)
    assert torch.equal(y, qmm.gemm("q4_0", wd, xd, n, k))
    y_ref, bound = oracle_mod.gemm_q4_0(w, xb, m, n, k)
    assert_within(y.cpu().numpy(), y_ref, bound, GEMM_REL, f"prefill {m}x{n}x{k}")


def test_prefill_static_scratch_column_chunks(qmm, oracle_mod):
    """K = 16384: the 64 MB scratch holds 2048 weight rows, so N = 5000 runs
    as three column chunks (2048, 2048, 904) written with the full row stride
    (600 tokens: 60 pair tiles, too many for a K split, so two phases)."""
    m, n, k = 600, 5000, 16384
    w, xb = synth.gemm_case(m, n, k, seed=77)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y = _prefill(qmm, wd, xd, m, n, k)
    assert torch.equal(y, qmm.gemm("q4_0", wd, xd, n, k))
    rng = np.random.default_rng(4)
    mi = rng.integers(0, m, 1500)
    ni = np.concatenate([rng.integers(0, n, 1496), [2047, 2048, 4095, 4999]])
    mi = np.concatenate([mi[:1496], [0, 1, m - 1, m - 1]])
    y_ref, bound = oracle_mod.gemm_q4_0_at(w, xb, m, n, k, mi, ni)
    assert_within(y.cpu().numpy()[mi, ni], y_ref, bound, GEMM_REL, "prefill chunks")


# ---- sparse last rounds run as 128-token half tiles ----

@pytest.mark.parametrize("m,n,k", [(1900, 2560, 512), (2048, 2560, 256)])
def test_two_phase_half_tile_tail(qmm, oracle_mod, m, n, k):
    """80 pair tiles over 76 pairs: the last 4 tiles run as 8 half tiles (ragged
    tokens in the first shape)."""
    w, xb = synth.gemm_case(m, n, k, seed=n + m)
    wd, xd = to_dev(w, torch), bf16_tensor(xb, torch)
    y2 = qmm.gemm("q4_0", wd, xd, n, k, workspace=_ws(qmm, n, k))
    y1 = qmm.gemm("q4_0", wd, xd, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(y2, y1)
    rng = np.random.default_rng(m)
    mi = np.concatenate([rng.integers(0, m, 3000), [m - 1, m - 1, 1792, 1920 % m]])
    ni = np.concatenate([rng.integers(0, n, 3000), [n - 1, 0, 2559, 2304]])
    y_ref, bound = oracle_mod.gemm_q4_0_at(w, xb, m, n, k, mi, ni)
    assert_within(y2.cpu().numpy()[mi, ni], y_ref, bound, GEMM_REL, f"half tail {m}x{n}x{k}")


def test_two_phase_geglu_half_tile_tail(qmm, oracle_mod):
    """GeGLU with 1280 features: 8 token blocks x 10 feature blocks = 80 tiles."""
    m, n, k = 2048, 1280, 512
    wg = synth.q4_0_weights(n, k, seed=8, stream=0)
    wu = synth.q4_0_weights(n, k, seed=8, stream=1)
    xb = synth.activations_bf16(m, k, seed=8, stream=2)
    a, b, xd = to_dev(wg, torch), to_dev(wu, torch), bf16_tensor(xb, torch)
    h2 = qmm.gemm_geglu_q4_0(a, b, xd, n, k, workspace=_ws(qmm, n, k, geglu=True))
    h1 = qmm.gemm_geglu_q4_0(a, b, xd, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(h2, h1)
    h_ref, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, _bf16_to_f32(xb)[1792:], m - 1792, n, k)
    assert_geglu_within(_bf16_to_f32(h2[1792:].cpu().numpy()), h_ref, g, u, bg, bu, "geglu tail",
                        rel=GEMM_REL, out_rel=2.0 ** -8)
