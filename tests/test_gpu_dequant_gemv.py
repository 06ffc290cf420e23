"""GPU parity: dequantization (bit-exact) and decode GEMV (1e-4 bound)
against the CPU oracle, through the C ABI."""
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


def _bits_equal_nan_class(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    if not np.array_equal(na, nb):
        return False
    return np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


def _special_q4_blocks():
    """Every nibble in both positions, for special and ordinary scales."""
    scales = [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00,
              0x3C00, 0xB800, 0x1234]
    blocks = []
    for d in scales:
        for v in range(16):
            qs = [(v | ((15 - v) << 4)) ^ (i * 0x11 & 0xFF) for i in range(16)]
            blocks.append([d & 0xFF, d >> 8] + qs)
    return np.array(blocks, dtype=np.uint8)


def _special_q8_blocks():
    scales = [0x0000, 0x8000, 0x0001, 0x7BFF, 0xFBFF, 0x7C00, 0x7E00, 0x3C00, 0xB555]
    blocks = []
    for d in scales:
        for start in range(0, 256, 32):
            blocks.append([d & 0xFF, d >> 8] + list(range(start, start + 32)))
    return np.array(blocks, dtype=np.uint8)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
def test_dequant_special_blocks_bit_exact(qmm, oracle_mod, fmt):
    blocks = _special_q4_blocks() if fmt == "q4_0" else _special_q8_blocks()
    n, k = blocks.shape[0], 32
    ref = (oracle_mod.dequant_q4_0 if fmt == "q4_0" else oracle_mod.dequant_q8_0)(blocks, n, k)
    got = qmm.dequant(fmt, to_dev(blocks, torch), n, k)
    torch.cuda.synchronize()
    assert _bits_equal_nan_class(got.cpu().numpy(), ref)


@pytest.mark.parametrize("fmt,n,k", [("q4_0", 37, 96), ("q4_0", 1000, 2048), ("q8_0", 129, 288),
                                     ("q8_0", 512, 2048), ("q4_0", 1, 32)])
def test_dequant_random_bit_exact(qmm, oracle_mod, fmt, n, k):
    case = synth.gemv_case(fmt, 1, n, k, seed=21)
    ref = (oracle_mod.dequant_q4_0 if fmt == "q4_0" else oracle_mod.dequant_q8_0)(case.w, n, k)
    got = qmm.dequant(fmt, to_dev(case.w, torch), n, k)
    torch.cuda.synchronize()
    assert _bits_equal_nan_class(got.cpu().numpy(), ref)


def test_dequant_unaligned_output(qmm, oracle_mod):
    n, k = 9, 64
    case = synth.gemv_case("q4_0", 1, n, k, seed=2)
    ref = oracle_mod.dequant_q4_0(case.w, n, k)
    buf = torch.empty(n * k + 1, dtype=torch.float32, device="cuda")
    out = buf[1:]
    qmm.qmm_dequant_q4_0(to_dev(case.w, torch), out.data_ptr(), n, k)
    torch.cuda.synchronize()
    assert _bits_equal_nan_class(out.cpu().numpy().reshape(n, k), ref)


def _run_gemv(qmm, fmt, case):
    w = to_dev(case.w, torch)
    x = to_dev(case.x, torch)
    y = qmm.gemv(fmt, w, x, case.n, case.k)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _oracle_gemv(oracle_mod, fmt, case):
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    return f(case.w, case.x, case.m, case.n, case.k)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("m", list(range(1, 17)))
def test_gemv_every_m(qmm, oracle_mod, fmt, m):
    # ragged rows (N % 32 != 0), several K chunks, small enough for the oracle
    case = synth.gemv_case(fmt, m, 203, 1280, seed=100 + m)
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    assert_within(_run_gemv(qmm, fmt, case), y_ref, bound, GEMV_REL, f"{fmt} m={m}")


@pytest.mark.parametrize("fmt,m,n,k", [
    ("q4_0", 1, 1, 256), ("q4_0", 3, 31, 256), ("q4_0", 2, 33, 512), ("q4_0", 1, 257, 8192),
    ("q4_0", 16, 64, 16384), ("q4_0", 5, 4000, 768), ("q8_0", 1, 1, 256), ("q8_0", 8, 257, 2048),
    ("q8_0", 16, 96, 8192), ("q4_0", 1, 512, 2048), ("q4_0", 4, 2048, 2048),
])
def test_gemv_shapes_streaming_path(qmm, oracle_mod, fmt, m, n, k):
    case = synth.gemv_case(fmt, m, n, k, seed=n + k)
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    assert_within(_run_gemv(qmm, fmt, case), y_ref, bound, GEMV_REL, f"{fmt} {m}x{n}x{k}")


@pytest.mark.parametrize("fmt,m,n,k", [("q4_0", 1, 7, 32), ("q4_0", 4, 65, 288), ("q8_0", 2, 33, 96),
                                       ("q8_0", 16, 40, 800)])
def test_gemv_bytewise_path_k_not_multiple_of_256(qmm, oracle_mod, fmt, m, n, k):
    case = synth.gemv_case(fmt, m, n, k, seed=3)
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    assert_within(_run_gemv(qmm, fmt, case), y_ref, bound, GEMV_REL, f"{fmt} {m}x{n}x{k}")


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
def test_gemv_unaligned_weights_take_bytewise_path(qmm, oracle_mod, fmt):
    m, n, k = 3, 45, 512
    case = synth.gemv_case(fmt, m, n, k, seed=8)
    raw = torch.zeros(case.w.size + 2, dtype=torch.uint8, device="cuda")
    raw[2:] = to_dev(case.w.reshape(-1), torch)
    x = to_dev(case.x, torch)
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    (qmm.qmm_gemv_q4_0 if fmt == "q4_0" else qmm.qmm_gemv_q8_0)(raw.data_ptr() + 2, x, y, m, n, k)
    torch.cuda.synchronize()
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    assert_within(y.cpu().numpy(), y_ref, bound, GEMV_REL, "unaligned w")


def test_gemv_degenerate_inputs(qmm):
    n, k = 70, 512
    # all nibbles 8 -> every weight zero; x arbitrary -> y == 0 exactly
    w = np.zeros((n, k // 32, 18), np.uint8)
    w[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    w[:, :, 2:] = 0x88
    x = synth.activations_f32(2, k, seed=1)
    y = qmm.gemv("q4_0", to_dev(w, torch), to_dev(x, torch), n, k)
    assert torch.count_nonzero(y).item() == 0
    # x == 0 -> y == 0
    case = synth.gemv_case("q8_0", 3, n, k, seed=1)
    y = qmm.gemv("q8_0", to_dev(case.w, torch), torch.zeros((3, k), device="cuda"), n, k)
    assert torch.count_nonzero(y).item() == 0


@pytest.mark.parametrize("m", [4, 16])
def test_gemv_deterministic(qmm, m):
    case = synth.gemv_case("q4_0", m, 2048, 2048, seed=5)
    w, x = to_dev(case.w, torch), to_dev(case.x, torch)
    a = qmm.gemv("q4_0", w, x, case.n, case.k)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = qmm.gemv("q4_0", w, x, case.n, case.k)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("cols", [[0, 17, 255, 256, 1023],
                                  # 12 rows of x: the row-pair form (M >= 11)
                                  [0, 1, 2, 3, 4, 15, 16, 19, 31, 511, 512, 1023]])
def test_gemv_one_hot_equals_dequant(qmm, cols):
    """x = e_c gives the dequantized column exactly (both on the GPU)."""
    n, k = 300, 1024
    case = synth.gemv_case("q4_0", 1, n, k, seed=6)
    w = to_dev(case.w, torch)
    x = torch.zeros((len(cols), k), device="cuda")
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    y = qmm.gemv("q4_0", w, x, n, k)
    deq = qmm.dequant("q4_0", w, n, k)
    for i, c in enumerate(cols):
        assert torch.equal(y[i], deq[:, c])


# ---- full-size workloads, in the launch configuration the benchmark times ----

def test_decode_layer_set_full(qmm, oracle_mod):
    for i, proj in enumerate(synth.DECODE_LAYER):
        case = synth.gemv_case("q4_0", 1, proj.n, proj.k, seed=0, stream=10 + i)
        y_ref, bound = _oracle_gemv(oracle_mod, "q4_0", case)
        assert_within(_run_gemv(qmm, "q4_0", case), y_ref, bound, GEMV_REL, proj.name)


@pytest.mark.parametrize("m", synth.BATCHED_M)
def test_batched_decode_full(qmm, oracle_mod, m):
    """Batched decode, both weight shapes: every output against the oracle."""
    for i, proj in enumerate(synth.BATCHED_SHAPES):
        case = synth.gemv_case("q4_0", m, proj.n, proj.k, seed=0, stream=30 + i)
        y_ref, bound = _oracle_gemv(oracle_mod, "q4_0", case)
        assert_within(_run_gemv(qmm, "q4_0", case), y_ref, bound, GEMV_REL, f"{proj.name} m={m}")


@pytest.mark.parametrize("m", synth.LM_HEAD_M)
def test_lm_head_q8_0_full(qmm, oracle_mod, m):
    """The Q8_0 LM head (262144 x 2048): every output against the oracle."""
    p = synth.LM_HEAD
    case = synth.gemv_case("q8_0", m, p.n, p.k, seed=0, stream=50)
    y = _run_gemv(qmm, "q8_0", case)
    y_ref, bound = _oracle_gemv(oracle_mod, "q8_0", case)
    assert_within(y, y_ref, bound, GEMV_REL, f"lm_head m={m}")


def test_timeout_path_reports_and_context_survives(qmm):
    qmm.qmm_get_device_error()  # clear
    qmm.qmm_selftest_wait_timeout(2_000_000)  # 2 ms
    assert qmm.qmm_get_device_error() == qmm.QMM_ERR_TIMEOUT
    assert qmm.qmm_get_device_error() == qmm.QMM_OK
    # the context still works
    case = synth.gemv_case("q4_0", 1, 64, 256, seed=1)
    y = qmm.gemv("q4_0", to_dev(case.w, torch), to_dev(case.x, torch), 64, 256)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()


# ---- grouped GEMV: several weight matrices sharing x in one launch ----

@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("m", [1, 2, 5, 16])
def test_gemv_multi_matches_oracle(qmm, oracle_mod, fmt, m):
    k = 2048
    ns = [2048, 512, 512] if fmt == "q4_0" else [1000, 96]
    x = synth.activations_f32(m, k, seed=60 + m)
    ws = [(synth.q4_0_weights if fmt == "q4_0" else synth.q8_0_weights)(n, k, seed=61, stream=i)
          for i, n in enumerate(ns)]
    xd = to_dev(x, torch)
    ys = [torch.empty((m, n), dtype=torch.float32, device="cuda") for n in ns]
    outs = [(to_dev(w, torch), y, n) for w, y, n in zip(ws, ys, ns)]
    (qmm.qmm_gemv_q4_0_multi if fmt == "q4_0" else qmm.qmm_gemv_q8_0_multi)(outs, xd, m, k)
    torch.cuda.synchronize()
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    for w, y, n in zip(ws, ys, ns):
        y_ref, bound = f(w, x, m, n, k)
        assert_within(y.cpu().numpy(), y_ref, bound, GEMV_REL, f"multi {fmt} m={m} n={n}")


def test_gemv_multi_decode_qkv_and_gate_up_full(qmm, oracle_mod):
    """The decode layer's grouped calls: q+k+v and gate+up, at full size."""
    k = 2048
    x = synth.activations_f32(1, k, seed=70)
    xd = to_dev(x, torch)
    for group in (("q", "k", "v"), ("gate", "up")):
        projs = [p for p in synth.DECODE_LAYER if p.name in group]
        ws = [synth.q4_0_weights(p.n, p.k, seed=71, stream=i) for i, p in enumerate(projs)]
        ys = [torch.empty((1, p.n), dtype=torch.float32, device="cuda") for p in projs]
        qmm.qmm_gemv_q4_0_multi([(to_dev(w, torch), y, p.n) for w, y, p in zip(ws, ys, projs)], xd, 1, k)
        torch.cuda.synchronize()
        for w, y, p in zip(ws, ys, projs):
            y_ref, bound = oracle_mod.gemv_q4_0(w, x, 1, p.n, k)
            assert_within(y.cpu().numpy(), y_ref, bound, GEMV_REL, f"multi {p.name}")


def test_gemv_multi_rejects_overlap_and_count(qmm):
    k, n = 256, 64
    w = torch.zeros(n * (k // 32) * 18, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, k), device="cuda")
    y = torch.empty((1, 2 * n), device="cuda")
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_gemv_q4_0_multi([(w, y, n), (w, y.view(-1)[8:], n)], x, 1, k)  # outputs overlap
    assert e.value.status == qmm.QMM_ERR_UNSUPPORTED
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_gemv_q4_0_multi([(w, y, n)] * 5, x, 1, k)
    assert e.value.status == qmm.QMM_ERR_SHAPE


# ---- M = 1, K % 2048 == 0: the row-balanced kernel (one CTA per SM, whole rows) ----

@pytest.mark.parametrize("n,k", [(1, 2048), (100, 2048), (151, 2048), (152, 2048), (153, 2048),
                                 (1000, 2048), (3001, 4096), (777, 8192), (300, 16384),
                                 (20000, 2048), (22000, 2048)])
def test_gemv_m1_row_balanced_shapes(qmm, oracle_mod, n, k):
    # ragged and tiny N around the SM count, K in 1..8 segments of 2048, and
    # N just inside / outside the shared-memory budget (the latter falls back
    # to the streaming kernel)
    case = synth.gemv_case("q4_0", 1, n, k, seed=n * 7 + k)
    if n * k > 8_000_000:
        rng = np.random.default_rng(n)
        ni = rng.integers(0, n, 4000)
        mi = np.zeros_like(ni)
        y_ref, bound = oracle_mod.gemv_q4_0_at(case.w, case.x, 1, n, k, mi, ni)
        assert_within(_run_gemv(qmm, "q4_0", case)[mi, ni], y_ref, bound, GEMV_REL, f"1x{n}x{k}")
    else:
        y_ref, bound = _oracle_gemv(oracle_mod, "q4_0", case)
        assert_within(_run_gemv(qmm, "q4_0", case), y_ref, bound, GEMV_REL, f"1x{n}x{k}")


@pytest.mark.parametrize("k,ns", [(2048, [5, 300, 1500, 7]), (8192, [100, 60]), (4096, [1, 151, 2])])
def test_gemv_m1_multi_rows_straddle_ctas(qmm, oracle_mod, k, ns):
    """Grouped problems whose boundaries fall inside a CTA's row range."""
    x = synth.activations_f32(1, k, seed=80)
    ws = [synth.q4_0_weights(n, k, seed=81, stream=i) for i, n in enumerate(ns)]
    ys = [torch.full((1, n), float("nan"), dtype=torch.float32, device="cuda") for n in ns]
    qmm.qmm_gemv_q4_0_multi([(to_dev(w, torch), y, n) for w, y, n in zip(ws, ys, ns)],
                            to_dev(x, torch), 1, k)
    torch.cuda.synchronize()
    for w, y, n in zip(ws, ys, ns):
        y_ref, bound = oracle_mod.gemv_q4_0(w, x, 1, n, k)
        assert_within(y.cpu().numpy(), y_ref, bound, GEMV_REL, f"multi k={k} n={n}")


def test_gemv_m1_one_hot_and_determinism(qmm):
    """x = e_c gives the dequantized column exactly; repeated calls are bitwise equal."""
    n, k = 1000, 4096
    case = synth.gemv_case("q4_0", 1, n, k, seed=9)
    w = to_dev(case.w, torch)
    deq = qmm.dequant("q4_0", w, n, k)
    for c in (0, 63, 64, 2047, 2048, 4095):
        x = torch.zeros((1, k), device="cuda")
        x[0, c] = 1.0
        y = qmm.gemv("q4_0", w, x, n, k)
        assert torch.equal(y[0], deq[:, c]), c
    x = to_dev(case.x, torch)
    a = qmm.gemv("q4_0", w, x, n, k)
    b = qmm.gemv("q4_0", w, x, n, k)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("fmt,m,n,k", [("q4_0", 16, 40, 65536), ("q8_0", 8, 33, 32768),
                                       ("q4_0", 10, 70, 32768)])
def test_gemv_very_large_k_falls_back_correctly(qmm, oracle_mod, fmt, m, n, k):
    """Activation slices too large for shared memory at any cluster split take
    the byte-wise kernel: still correct, never an error status."""
    case = synth.gemv_case(fmt, m, n, k, seed=m + n)
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    assert_within(_run_gemv(qmm, fmt, case), y_ref, bound, GEMV_REL, f"{fmt} {m}x{n}x{k}")


@pytest.mark.parametrize("fmt,m,n,k", [("q8_0", 8, 300, 8192), ("q8_0", 9, 70, 16384),
                                       ("q4_0", 6, 1000, 2048), ("q4_0", 10, 257, 4096)])
def test_gemv_wide_m_two_rows_per_lane_and_its_fallback(qmm, oracle_mod, fmt, m, n, k):
    """M = 5..10 uses two weight rows per lane; shapes whose shared memory does
    not fit that form fall back to one row per lane (Q8_0 at K = 16384)."""
    case = synth.gemv_case(fmt, m, n, k, seed=m * 13 + n)
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    assert_within(_run_gemv(qmm, fmt, case), y_ref, bound, GEMV_REL, f"{fmt} {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(11, 200, 2048), (13, 1000, 4096), (16, 70, 8192), (11, 3000, 256),
                                   (16, 130, 16384), (11, 16384, 16384), (16, 130, 32768),
                                   (11, 256, 18432)])
def test_gemv_row_pairs_and_their_fallback(qmm, oracle_mod, m, n, k):
    """Q4_0 at M >= 11 packs two weight rows into each FMA with the block scale
    folded into the weights: ragged 64-row tiles, cluster splits (up to 8 x 8
    K parts at 130 x 16384), several tiles per launch, and 16384 x 16384, where
    each accumulator sums the most products the form allows (8 chunks, 1024
    per lane).  The last two shapes leave the row-pair form: at 130 x 32768 its
    activation slice does not fit shared memory; at 256 x 18432 (72 chunks, at
    most 8 K parts) a lane's share would be 1152 products."""
    case = synth.gemv_case("q4_0", m, n, k, seed=m * 7 + n)
    y_ref, bound = _oracle_gemv(oracle_mod, "q4_0", case)
    assert_within(_run_gemv(qmm, "q4_0", case), y_ref, bound, GEMV_REL, f"q4_0 {m}x{n}x{k}")


@pytest.mark.parametrize("fmt,m,n,k", [("q4_0", 1, 80000, 256), ("q4_0", 2, 100003, 512),
                                       ("q4_0", 4, 90000, 2048), ("q4_0", 3, 78000, 1280),
                                       ("q8_0", 1, 40000, 2048), ("q8_0", 2, 50001, 768),
                                       ("q4_0", 6, 80000, 1280), ("q4_0", 9, 90001, 512),
                                       ("q8_0", 8, 40000, 2048), ("q4_0", 1, 77000, 512)])
def test_gemv_persistent_form(qmm, oracle_mod, fmt, m, n, k):
    """Large single matrices at M <= 10 run one CTA per SM over an even share of
    whole tiles, their warps splitting the units so that some tiles are shared
    by two warps (K = 512, 1280, 768, 2048: several chunks per tile) and added
    after a CTA barrier; ragged N (100003, 50001, 90001); M = 6, 8, 9 use the
    per-block loop of wide M; 77000 x 512 has too few tiles for every warp and
    takes the streaming form."""
    case = synth.gemv_case(fmt, m, n, k, seed=n % 1000 + k)
    y_ref, bound = _oracle_gemv(oracle_mod, fmt, case)
    y = _run_gemv(qmm, fmt, case)
    assert qmm.qmm_get_device_error() == 0
    assert_within(y, y_ref, bound, GEMV_REL, f"{fmt} {m}x{n}x{k}")


def test_gemv_persistent_form_deterministic(qmm):
    case = synth.gemv_case("q4_0", 2, 100003, 1280, seed=11)
    w, x = to_dev(case.w, torch), to_dev(case.x, torch)
    a = qmm.gemv("q4_0", w, x, case.n, case.k)
    b = qmm.gemv("q4_0", w, x, case.n, case.k)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("n,k", [(2048, 8192), (2000, 8192), (1000, 16384), (520, 32768), (3000, 4096)])
def test_gemv_m1_long_k_two_lanes(qmm, oracle_mod, n, k):
    """M = 1 with few rows and a long K: two lanes per row where that needs a
    smaller cluster split than one lane per row (2048 x 8192: clusters of 2
    instead of 4; ragged rows at 2000 and 520; K = 16384 and 32768), one lane
    per row where both need the same (3000 x 4096).  Every output against
    the oracle, and the same bits on a second call."""
    case = synth.gemv_case("q4_0", 1, n, k, seed=n + k)
    w, x = to_dev(case.w, torch), to_dev(case.x, torch)
    a = qmm.gemv("q4_0", w, x, n, k)
    b = qmm.gemv("q4_0", w, x, n, k)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    y_ref, bound = _oracle_gemv(oracle_mod, "q4_0", case)
    assert_within(a.cpu().numpy(), y_ref, bound, GEMV_REL, f"q4_0 1x{n}x{k}")
