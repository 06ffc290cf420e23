"""Pins for the CPU oracle: values fixed by the block formats and by the
mathematics of the product, checked without trusting the oracle itself.

The formats are GGUF Q4_0 and Q8_0, the two block formats whose dispatches
are counted in "Add generated quant-kernel JIT and accelerate Gemma4, BGE-M3,
and GLiNER2", section "Validation" (342 Q4_0 and one Q8_0 per decode token).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from block_quantized_matmul_gguf_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gguf_blocks.json")


def _hexbytes(s):
    return np.frombuffer(bytes.fromhex(s.replace(" ", "")), dtype=np.uint8)


def _expect(vals):
    return np.array([float(v) for v in vals], dtype=np.float64)


def q4_block(d_bits, qs):
    return np.array([d_bits & 0xFF, d_bits >> 8] + list(qs), dtype=np.uint8)


def q8_block(d_bits, q):
    return np.array([d_bits & 0xFF, d_bits >> 8] + [v & 0xFF for v in q], dtype=np.uint8)


def f16bits(v):
    return int(np.array(v, dtype=np.float16).view(np.uint16))


# ---------------------------------------------------------------- binary16 / bf16

def test_fp16_decode_exhaustive_against_numpy(oracle_mod):
    lib = oracle_mod._load()
    bits = np.arange(65536, dtype=np.uint32)
    ours = np.array([lib.qmm_oracle_fp16_to_f64(int(b)) for b in bits])
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24),
    (0x0400, 2.0 ** -14), (0x7BFF, 65504.0), (0xC000, -2.0), (0x3555, 0.25 * (1 + 0x155 / 1024)),
])
def test_fp16_spot_values(oracle_mod, bits, value):
    assert oracle_mod.fp16_to_f64(bits) == value


def test_fp16_specials(oracle_mod):
    assert oracle_mod.fp16_to_f64(0x7C00) == math.inf
    assert oracle_mod.fp16_to_f64(0xFC00) == -math.inf
    assert math.isnan(oracle_mod.fp16_to_f64(0x7E00))
    z = oracle_mod.fp16_to_f64(0x8000)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


def test_bf16_decode_exhaustive_against_torch(oracle_mod):
    lib = oracle_mod._load()
    bits = np.arange(65536, dtype=np.int64)
    ours = np.array([lib.qmm_oracle_bf16_to_f64(int(b)) for b in bits])
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ---------------------------------------------------------------- block formats

def test_golden_blocks(oracle_mod):
    data = json.load(open(GOLDEN))
    for blk in data["blocks"]:
        raw = _hexbytes(blk["hex"])
        exp = _expect(blk["expect"])
        if blk["format"] == "q4_0":
            assert raw.size == 18, blk["name"]
            got = oracle_mod.dequant_q4_0(raw, 1, 32)[0].astype(np.float64)
        else:
            assert raw.size == 34, blk["name"]
            got = oracle_mod.dequant_q8_0(raw, 1, 32)[0].astype(np.float64)
        assert np.array_equal(got, exp), blk["name"]
        assert np.array_equal(np.signbit(got), np.signbit(exp)), blk["name"]


def test_golden_gemv(oracle_mod):
    data = json.load(open(GOLDEN))
    for case in data["gemv"]:
        raw = _hexbytes(case["row_hex"])
        x = np.ones((case["m"], case["k"]), dtype=np.float32)
        y, bound = oracle_mod.gemv_q4_0(raw, x, case["m"], case["n"], case["k"])
        assert y[0, 0] == case["expect_y"]
        assert bound[0, 0] == case["expect_bound"]


@pytest.mark.parametrize("d", [1.0, 0.5, -2.0, 0.0078125])
def test_q4_0_every_nibble_every_position(oracle_mod, d):
    """Nibble v at weight position p gives (v-8)*d there and zero elsewhere.

    Pins the nibble order: position p < 16 is the low nibble of byte p,
    position p >= 16 the high nibble of byte p-16."""
    db = f16bits(d)
    blocks, expect = [], []
    for p in range(32):
        for v in range(16):
            qs = [0x88] * 16
            if p < 16:
                qs[p] = (qs[p] & 0xF0) | v
            else:
                qs[p - 16] = (qs[p - 16] & 0x0F) | (v << 4)
            blocks.append(q4_block(db, qs))
            e = np.zeros(32)
            e[p] = (v - 8) * d
            expect.append(e)
    got = oracle_mod.dequant_q4_0(np.concatenate(blocks), len(blocks), 32)
    assert np.array_equal(got.astype(np.float64), np.array(expect))


def test_q4_0_format_checks(oracle_mod):
    d = 0.013
    db = f16bits(d)
    dd = float(np.float16(d))
    for pos_byte, shift, idx in [(3, 0, 3), (3, 4, 19)]:
        for v, want in [(0, -8 * dd), (8, 0.0), (15, 7 * dd)]:
            qs = [0x88] * 16
            # the other nibble of the byte stays 8 (weight 0)
            qs[pos_byte] = (0x80 | v) if shift == 0 else ((v << 4) | 0x08)
            w = oracle_mod.dequant_q4_0(q4_block(db, qs), 1, 32)[0]
            assert w[idx] == np.float32(want)
    # byte 0xF0 at j: w[j] = -8d, w[j+16] = 7d
    qs = [0x88] * 16
    qs[5] = 0xF0
    w = oracle_mod.dequant_q4_0(q4_block(db, qs), 1, 32)[0]
    assert w[5] == np.float32(-8 * dd) and w[21] == np.float32(7 * dd)
    # d = 0 gives all zeros, whatever the nibbles
    rng = np.random.default_rng(1)
    qs = list(rng.integers(0, 256, 16))
    w = oracle_mod.dequant_q4_0(q4_block(0x0000, qs), 1, 32)[0]
    assert np.all(w == 0.0)


def test_q4_0_zero_sign_and_nonfinite(oracle_mod):
    qs = [0x88] * 16
    qs[0] = 0x80  # low nibble 0 (w[0] = -8d), high nibble 8 (w[16] = 0*d)
    w = oracle_mod.dequant_q4_0(q4_block(f16bits(-1.0), qs), 1, 32)[0]
    assert w[0] == 8.0 and w[16] == 0.0 and np.signbit(w[16])
    w = oracle_mod.dequant_q4_0(q4_block(0x7C00, qs), 1, 32)[0]  # d = +inf
    assert w[0] == -np.inf and np.isnan(w[16])
    w = oracle_mod.dequant_q4_0(q4_block(0x7E00, qs), 1, 32)[0]  # d = NaN
    assert np.all(np.isnan(w))


def test_q8_0_every_byte(oracle_mod):
    for d in (1.0, 0.5, -0.25):
        db = f16bits(d)
        blocks = [q8_block(db, list(range(32 * i, 32 * i + 32))) for i in range(8)]
        got = oracle_mod.dequant_q8_0(np.concatenate(blocks), 8, 32).reshape(-1)
        vals = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
        assert np.array_equal(got.astype(np.float64), vals * d)


def test_q8_0_format_checks(oracle_mod):
    w = oracle_mod.dequant_q8_0(q8_block(f16bits(1.0), [127, -127, 0, -128] + [0] * 28), 1, 32)[0]
    assert list(w[:4]) == [127.0, -127.0, 0.0, -128.0]


def test_dequant_row_major_layout(oracle_mod):
    """Block b of row n sits at byte (n*(K/32)+b)*18: give each block its own
    scale and check where each scale lands."""
    n, k = 3, 96
    blocks = []
    for r in range(n):
        for b in range(k // 32):
            blocks.append(q4_block(f16bits(float(1 + 10 * r + b)), [0x99] * 16))
    w = oracle_mod.dequant_q4_0(np.concatenate(blocks), n, k)
    for r in range(n):
        for b in range(k // 32):
            assert np.all(w[r, 32 * b:32 * b + 32] == float(1 + 10 * r + b))


# ---------------------------------------------------------------- products

def _dense_by_offsets(w_bytes, n, k, fmt):
    """Dense W built weight by weight from byte offsets (independent of the
    oracle's block walk): Q4_0 weight (n, k) is nibble (k%32 >= 16) of byte
    2 + (k%32)%16 of block n*(K/32) + k/32; the scale is decoded by numpy."""
    bb = 18 if fmt == "q4_0" else 34
    wb = np.asarray(w_bytes, dtype=np.uint8).reshape(-1)
    out = np.zeros((n, k))
    for r in range(n):
        for c in range(k):
            base = (r * (k // 32) + c // 32) * bb
            d = float(wb[base:base + 2].view(np.float16)[0])
            j = c % 32
            if fmt == "q4_0":
                byte = int(wb[base + 2 + j % 16])
                nib = (byte >> 4) if j >= 16 else (byte & 15)
                out[r, c] = (nib - 8) * d
            else:
                out[r, c] = float(wb[base + 2 + j:base + 3 + j].view(np.int8)[0]) * d
    return out


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
def test_brute_force_2x64(oracle_mod, fmt):
    """N=2, K=64, M=2, integer-valued x and power-of-two d: every product and
    sum is exact, so the oracle must equal an independent double loop."""
    rng = np.random.default_rng(7)
    n, k, m = 2, 64, 2
    blocks = []
    for _ in range(n * k // 32):
        d = f16bits(float(2.0 ** rng.integers(-6, 3)) * (1 if rng.random() < 0.5 else -1))
        if fmt == "q4_0":
            blocks.append(q4_block(d, list(rng.integers(0, 256, 16))))
        else:
            blocks.append(q8_block(d, list(rng.integers(-128, 128, 32))))
    w = np.concatenate(blocks)
    x = rng.integers(-9, 10, size=(m, k)).astype(np.float32)
    dense = _dense_by_offsets(w, n, k, fmt)
    y_ref = np.zeros((m, n))
    b_ref = np.zeros((m, n))
    for i in range(m):
        for r in range(n):
            for c in range(k):
                y_ref[i, r] += float(x[i, c]) * dense[r, c]
                b_ref[i, r] += abs(float(x[i, c]) * dense[r, c])
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    y, bound = f(w, x, m, n, k)
    assert np.array_equal(y, y_ref)
    assert np.array_equal(bound, b_ref)
    deq = oracle_mod.dequant_q4_0(w, n, k) if fmt == "q4_0" else oracle_mod.dequant_q8_0(w, n, k)
    assert np.array_equal(deq.astype(np.float64), dense)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
def test_one_hot_columns(oracle_mod, fmt):
    """x = e_c gives y[n] = w[n][c] exactly: ties the product to the (pinned)
    dequantization and catches a transposed operand (N != K)."""
    n, k = 5, 96
    w = synth.q4_0_weights(n, k, 3) if fmt == "q4_0" else synth.q8_0_weights(n, k, 3)
    deq = oracle_mod.dequant_q4_0(w, n, k) if fmt == "q4_0" else oracle_mod.dequant_q8_0(w, n, k)
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    cols = [0, 1, 15, 16, 31, 32, 63, 95]
    x = np.zeros((len(cols), k), dtype=np.float32)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    y, bound = f(w, x, len(cols), n, k)
    for i, c in enumerate(cols):
        assert np.array_equal(y[i], deq[:, c].astype(np.float64))
        assert np.array_equal(bound[i], np.abs(deq[:, c]).astype(np.float64))


def test_linearity_power_of_two(oracle_mod):
    """y(a*x1 + b*x2) = a*y(x1) + b*y(x2) for a, b powers of two and
    integer-valued x, d powers of two (all sums exact)."""
    rng = np.random.default_rng(11)
    n, k = 7, 128
    blocks = [q4_block(f16bits(float(2.0 ** rng.integers(-4, 2))), list(rng.integers(0, 256, 16)))
              for _ in range(n * k // 32)]
    w = np.concatenate(blocks)
    x1 = rng.integers(-50, 50, size=(1, k)).astype(np.float32)
    x2 = rng.integers(-50, 50, size=(1, k)).astype(np.float32)
    a, b = 4.0, -0.5
    y1, _ = oracle_mod.gemv_q4_0(w, x1, 1, n, k)
    y2, _ = oracle_mod.gemv_q4_0(w, x2, 1, n, k)
    y3, _ = oracle_mod.gemv_q4_0(w, (a * x1 + b * x2).astype(np.float32), 1, n, k)
    assert np.array_equal(y3, a * y1 + b * y2)


@pytest.mark.parametrize("c", [0, 3, 8, 12, 15])
def test_closed_form_constant_nibbles(oracle_mod, c):
    """x = 1 and every nibble = c: y[n] = K*(c-8)*d."""
    n, k, d = 3, 256, 0.0625
    blocks = [q4_block(f16bits(d), [c | (c << 4)] * 16) for _ in range(n * k // 32)]
    y, bound = oracle_mod.gemv_q4_0(np.concatenate(blocks), np.ones((2, k), np.float32), 2, n, k)
    assert np.all(y == k * (c - 8) * d)
    assert np.all(bound == k * abs(c - 8) * d)


@pytest.mark.parametrize("fmt,m,n,k", [("q4_0", 3, 17, 160), ("q8_0", 2, 9, 256), ("q4_0", 1, 64, 1024)])
def test_against_numpy_matmul(oracle_mod, fmt, m, n, k):
    """Random inputs: the oracle equals numpy's float64 matmul of the pinned
    dequantization to within binary64 summation rounding."""
    case = synth.gemv_case(fmt, m, n, k, seed=5)
    deq = (oracle_mod.dequant_q4_0 if fmt == "q4_0" else oracle_mod.dequant_q8_0)(case.w, n, k)
    ref = case.x.astype(np.float64) @ deq.astype(np.float64).T
    absref = np.abs(case.x.astype(np.float64)) @ np.abs(deq.astype(np.float64)).T
    f = oracle_mod.gemv_q4_0 if fmt == "q4_0" else oracle_mod.gemv_q8_0
    y, bound = f(case.w, case.x, m, n, k)
    assert np.all(np.abs(y - ref) <= 1e-12 * absref)
    assert np.allclose(bound, absref, rtol=1e-12, atol=0)
    assert np.all(bound >= np.abs(y))


def test_gemm_bf16_against_numpy(oracle_mod):
    m, n, k = 6, 11, 192
    w, xb = synth.gemm_case(m, n, k, seed=9)
    xv = torch.from_numpy(xb.astype(np.int16)).view(torch.bfloat16).double().numpy()
    deq = oracle_mod.dequant_q4_0(w, n, k).astype(np.float64)
    y, bound = oracle_mod.gemm_q4_0(w, xb, m, n, k)
    ref = xv @ deq.T
    absref = np.abs(xv) @ np.abs(deq).T
    assert np.all(np.abs(y - ref) <= 1e-12 * absref)
    assert np.allclose(bound, absref, rtol=1e-12, atol=0)


def test_gemm_one_hot(oracle_mod):
    m, n, k = 3, 4, 64
    w = synth.q4_0_weights(n, k, 2)
    deq = oracle_mod.dequant_q4_0(w, n, k)
    x = np.zeros((m, k), dtype=np.uint16)
    cols = [2, 33, 63]
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80  # bf16 1.0
    y, _ = oracle_mod.gemm_q4_0(w, x, m, n, k)
    for i, c in enumerate(cols):
        assert np.array_equal(y[i], deq[:, c].astype(np.float64))


def test_sampled_outputs_match_full(oracle_mod):
    m, n, k = 3, 40, 256
    case = synth.gemv_case("q4_0", m, n, k, seed=4)
    y, bound = oracle_mod.gemv_q4_0(case.w, case.x, m, n, k)
    mi = np.array([0, 2, 1, 2])
    ni = np.array([0, 39, 17, 5])
    ys, bs = oracle_mod.gemv_q4_0_at(case.w, case.x, m, n, k, mi, ni)
    assert np.array_equal(ys, y[mi, ni]) and np.array_equal(bs, bound[mi, ni])
    case8 = synth.gemv_case("q8_0", m, n, k, seed=4)
    y8, b8 = oracle_mod.gemv_q8_0(case8.w, case8.x, m, n, k)
    ys8, bs8 = oracle_mod.gemv_q8_0_at(case8.w, case8.x, m, n, k, mi, ni)
    assert np.array_equal(ys8, y8[mi, ni]) and np.array_equal(bs8, b8[mi, ni])
    w, xb = synth.gemm_case(m, n, k, seed=4)
    yg, bg = oracle_mod.gemm_q4_0(w, xb, m, n, k)
    ysg, bsg = oracle_mod.gemm_q4_0_at(w, xb, m, n, k, mi, ni)
    assert np.array_equal(ysg, yg[mi, ni]) and np.array_equal(bsg, bg[mi, ni])
    wu = synth.q4_0_weights(n, k, seed=5)
    full = oracle_mod.geglu_q4_0(case.w, wu, case.x, m, n, k)
    at = oracle_mod.geglu_q4_0_at(case.w, wu, case.x, m, n, k, mi, ni)
    for a, f in zip(at, full):
        assert np.array_equal(a, f[mi, ni])


# ---------------------------------------------------------------- tolerance sanity

def within(y, y_ref, bound, rel):
    return np.abs(np.asarray(y, np.float64) - y_ref) <= rel * bound + 1e-6


def test_fp32_accumulation_meets_gemv_bound(oracle_mod):
    """The 1e-4 GEMV bound is attainable: a plain sequential fp32 sum of the
    exact products passes it; one flipped nibble fails it."""
    m, n, k = 2, 64, 8192
    case = synth.gemv_case("q4_0", m, n, k, seed=12)
    y_ref, bound = oracle_mod.gemv_q4_0(case.w, case.x, m, n, k)
    deq = oracle_mod.dequant_q4_0(case.w, n, k)
    y32 = np.zeros((m, n), dtype=np.float32)
    for c in range(k):  # strictly sequential fp32 accumulation
        y32 += case.x[:, c:c + 1] * deq[:, c][None, :]
    assert np.all(within(y32, y_ref, bound, 1e-4))
    bad = case.w.copy().reshape(-1)
    # move weight 0 of row 0 to the opposite end of the nibble range
    bad[2] = (bad[2] & 0xF0) | (0x0 if (case.w.reshape(-1)[2] & 0xF) >= 8 else 0xF)
    y_bad, _ = oracle_mod.gemv_q4_0(bad, case.x, m, n, k)
    assert not np.all(within(y_bad, y_ref, bound, 1e-4))


# ---------------------------------------------------------------- generator

def test_generator_deterministic_and_in_range():
    a = synth.q4_0_weights(16, 256, seed=0, stream=3)
    b = synth.q4_0_weights(16, 256, seed=0, stream=3)
    c = synth.q4_0_weights(16, 256, seed=1, stream=3)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    d = a.reshape(-1, 18)[:, :2].copy().view(np.float16).astype(np.float64)
    assert d.min() >= 0.001 - 1e-6 and d.max() <= 0.02 + 1e-5
    q = synth.q8_0_weights(64, 512, seed=0)
    qv = q.reshape(-1, 34)[:, 2:].view(np.int8)
    assert qv.min() >= -127 and qv.max() <= 127
    hist = np.bincount(qv.reshape(-1).astype(np.int64) + 127, minlength=255)
    assert hist.min() > 0
    x = synth.activations_f32(4, 4096, seed=0)
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05
    nib = np.concatenate([a.reshape(-1, 18)[:, 2:] & 15, a.reshape(-1, 18)[:, 2:] >> 4]).reshape(-1)
    assert np.bincount(nib, minlength=16).min() > 0


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.005859375, 1.01171875, -3.3e-3], dtype=np.float32)
    ours = synth.f32_to_bf16_bits(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(ours, ref)
    big = synth.activations_f32(1, 1 << 16, seed=3).reshape(-1)
    ref = torch.from_numpy(big).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(big), ref)


# ---- GeGLU feed-forward input: h = gelu_tanh(x.Wg^T) * (x.Wu^T) ----

def _one_block_rows(nibbles, scales):
    """Q4_0 rows of one block each: weight 0 (low nibble of qs[0]) = nibbles[i],
    every other weight nibble 8 (zero); d = scales[i] (rounded to binary16)."""
    rows = []
    for v, d in zip(nibbles, scales):
        blk = np.zeros(18, dtype=np.uint8)
        blk[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
        blk[2:] = 0x88
        blk[2] = 0x80 | v  # weight 0 = v, weight 16 = 8
        rows.append(blk)
    return np.stack(rows)


def test_geglu_activation_matches_torch_gelu_tanh(oracle_mod):
    """One-hot x = e_0 makes g = (v-8)*d and u = 1, so h = gelu(g): checked
    against torch's own float64 GELU (tanh form), an independent routine."""
    torch = pytest.importorskip("torch")
    vals, ds = [], []
    for d in (0.25, 1.0, 3.0, 100.0, 1e-3):
        for v in range(16):
            vals.append(v)
            ds.append(d)
    n, k = len(vals), 32
    wg = _one_block_rows(vals, ds)
    wu = _one_block_rows([9] * n, [1.0] * n)  # u = 1 exactly
    x = np.zeros((1, k), dtype=np.float32)
    x[0, 0] = 1.0
    h, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, x, 1, n, k)
    g_want = np.array([(v - 8) * float(np.float16(d)) for v, d in zip(vals, ds)])
    assert np.array_equal(g[0], g_want) and np.all(u == 1.0)
    want = torch.nn.functional.gelu(torch.from_numpy(g_want), approximate="tanh").numpy()
    np.testing.assert_allclose(h[0], want, rtol=1e-13, atol=1e-300)
    assert h[0][vals.index(8)] == 0.0          # gelu(0) = 0
    assert np.all(bg[0] == np.abs(g_want)) and np.all(bu[0] == 1.0)


def test_geglu_composes_the_pinned_products(oracle_mod):
    """h = gelu(g) * u with g, u the (pinned) GEMV of the gate and up weights:
    the activation is on the gate operand, and the product is elementwise."""
    torch = pytest.importorskip("torch")
    m, n, k = 3, 37, 256
    wg = synth.q4_0_weights(n, k, seed=11)
    wu = synth.q4_0_weights(n, k, seed=12)
    x = synth.activations_f32(m, k, seed=13)
    h, g, u, bg, bu = oracle_mod.geglu_q4_0(wg, wu, x, m, n, k)
    g_ref, bg_ref = oracle_mod.gemv_q4_0(wg, x, m, n, k)
    u_ref, bu_ref = oracle_mod.gemv_q4_0(wu, x, m, n, k)
    assert np.array_equal(g, g_ref) and np.array_equal(u, u_ref)
    assert np.array_equal(bg, bg_ref) and np.array_equal(bu, bu_ref)
    want = torch.nn.functional.gelu(torch.from_numpy(g_ref), approximate="tanh").numpy() * u_ref
    np.testing.assert_allclose(h, want, rtol=1e-13, atol=1e-300)
    # swapping the roles of gate and up gives a different result
    h_sw = oracle_mod.geglu_q4_0(wu, wg, x, m, n, k)[0]
    assert not np.allclose(h_sw, h, rtol=1e-3)
