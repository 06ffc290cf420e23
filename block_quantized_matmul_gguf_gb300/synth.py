"""Seeded synthetic inputs for the quantized matmul path.

This module only draws inputs.  It holds none of the method's arithmetic (no
dequantization, no dot product): it produces GGUF block bytes, fp32
activations and bf16 activation bit patterns that both the GPU library and the
CPU oracle consume unchanged.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator: draw i of stream (seed, stream) is mix64(key + (i+1) * GAMMA), with
key derived from seed and stream id.  Distributions:

* U[0,1): the top 53 bits of a draw times 2^-53.
* N(0,1): Box-Muller in binary64 on pairs (u1, u2), radius from 1-u1 so that
  log(0) never occurs; cos and sin of each pair give two values.
* binary16 scale d ~ U[lo, hi]: binary64 uniform rounded to nearest-even
  binary16 (numpy astype).
* Q4_0 nibble bytes: uniform bytes, i.e. two independent uniform nibbles.
* Q8_0 q ~ U{-127..127}: uniform bytes read as int8, with every -128
  redrawn from a follow-up stream until none is left.
* fp32 x: N(0,1) rounded to nearest-even binary32.
* bf16 X: N(0,1) rounded to binary32, then to nearest-even bfloat16.

The workloads below are the shapes of the Gemma4-style decode and prefill
products whose 342 Q4_0 and one Q8_0 dispatches per decode token are counted
in "Add generated quant-kernel JIT and accelerate Gemma4, BGE-M3, and GLiNER2",
section "Validation".
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

QK = 32
Q4_0_BYTES = 18
Q8_0_BYTES = 34

_CHUNK = 1 << 22  # draws generated per numpy pass (bounds peak host memory)


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of stream `stream` under `seed`."""
    return _mix64_int((seed + 1) * GAMMA) ^ _mix64_int((stream + 1) * 0xD1B54A32D192ED03)


def draws_u64(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Draws start .. start+count-1 of a stream, as uint64."""
    key = np.uint64(stream_key(seed, stream))
    out = np.empty(count, dtype=np.uint64)
    g = np.uint64(GAMMA)
    m1, m2 = np.uint64(_M1), np.uint64(_M2)
    s30, s27, s31 = np.uint64(30), np.uint64(27), np.uint64(31)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            z = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64) * g + key
            z = (z ^ (z >> s30)) * m1
            z = (z ^ (z >> s27)) * m2
            out[lo:hi] = z ^ (z >> s31)
    return out


def uniform01(seed: int, stream: int, count: int) -> np.ndarray:
    u = draws_u64(seed, stream, count)
    return (u >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))


def uniform_bytes(seed: int, stream: int, count: int) -> np.ndarray:
    words = draws_u64(seed, stream, (count + 7) // 8)
    return words.view(np.uint8)[:count].copy()


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """count N(0,1) values in binary64 (Box-Muller on consecutive draw pairs)."""
    pairs = (count + 1) // 2
    u = uniform01(seed, stream, 2 * pairs)
    r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
    theta = 2.0 * np.pi * u[1::2]
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(theta)
    z[1::2] = r * np.sin(theta)
    return z[:count]


def fp16_scales(seed: int, stream: int, count: int, lo: float, hi: float) -> np.ndarray:
    """binary16 bit patterns of d ~ U[lo, hi] (round to nearest even)."""
    u = uniform01(seed, stream, count)
    d = (lo + (hi - lo) * u).astype(np.float16)
    return d.view(np.uint16)


def _pack_blocks(d_bits: np.ndarray, payload: np.ndarray, block_bytes: int) -> np.ndarray:
    nblocks = d_bits.size
    out = np.empty((nblocks, block_bytes), dtype=np.uint8)
    out[:, 0] = (d_bits & 0xFF).astype(np.uint8)
    out[:, 1] = (d_bits >> 8).astype(np.uint8)
    out[:, 2:] = payload.reshape(nblocks, block_bytes - 2)
    return out


def q4_0_weights(n: int, k: int, seed: int = 0, stream: int = 0,
                 d_lo: float = 0.001, d_hi: float = 0.02) -> np.ndarray:
    """Q4_0 blocks of an n x k matrix: uint8 [n, k/32*18]."""
    if k % QK:
        raise ValueError("k must be a multiple of 32")
    nb = n * (k // QK)
    d = fp16_scales(seed, 2 * stream, nb, d_lo, d_hi)
    qs = uniform_bytes(seed, 2 * stream + 1, nb * 16)
    return _pack_blocks(d, qs, Q4_0_BYTES).reshape(n, (k // QK) * Q4_0_BYTES)


def q8_0_weights(n: int, k: int, seed: int = 0, stream: int = 0,
                 d_lo: float = 1e-4, d_hi: float = 4e-3) -> np.ndarray:
    """Q8_0 blocks of an n x k matrix, q ~ U{-127..127}: uint8 [n, k/32*34]."""
    if k % QK:
        raise ValueError("k must be a multiple of 32")
    nb = n * (k // QK)
    d = fp16_scales(seed, 2 * stream, nb, d_lo, d_hi)
    q = uniform_bytes(seed, 2 * stream + 1, nb * 32)
    redraw = 0
    bad = np.flatnonzero(q == 0x80)
    while bad.size:
        redraw += 1
        # follow-up streams live far above the ids used for first draws
        fresh = uniform_bytes(seed, (1 << 40) + 64 * stream + redraw, bad.size)
        q[bad] = fresh
        bad = bad[fresh == 0x80]
    return _pack_blocks(d, q, Q8_0_BYTES).reshape(n, (k // QK) * Q8_0_BYTES)


def activations_f32(m: int, k: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """fp32 [m, k] with values N(0,1)."""
    return normal(seed, stream, m * k).astype(np.float32).reshape(m, k)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to nearest-even bfloat16, returned as uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def activations_bf16(m: int, k: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """bf16 bit patterns uint16 [m, k] with values N(0,1)."""
    return f32_to_bf16_bits(activations_f32(m, k, seed, stream))


# ---------------------------------------------------------------------------
# Workloads.  W is N rows x K columns; a projection "a->b" has K=a, N=b.

@dataclass(frozen=True)
class Projection:
    name: str
    n: int
    k: int


DECODE_LAYER = (
    Projection("q", 2048, 2048),
    Projection("k", 512, 2048),
    Projection("v", 512, 2048),
    Projection("o", 2048, 2048),
    Projection("gate", 8192, 2048),
    Projection("up", 8192, 2048),
    Projection("down", 2048, 8192),
)

SINGLE_SMALL = Projection("small", 256, 1024)
BATCHED_SHAPES = (Projection("wide", 8192, 2048), Projection("tall", 2048, 8192))
BATCHED_M = (2, 4, 8, 16)
LM_HEAD = Projection("lm_head", 262144, 2048)
LM_HEAD_M = (1, 8)
PREFILL_M = 2048
PREFILL_SHAPES = (Projection("wide", 8192, 2048), Projection("tall", 2048, 8192))
SHORT_PROMPT_M = 256  # the shortest prefill the GEMM path takes (M >= 256)


def q4_0_bytes(n: int, k: int) -> int:
    return n * (k // QK) * Q4_0_BYTES


def q8_0_bytes(n: int, k: int) -> int:
    return n * (k // QK) * Q8_0_BYTES


@dataclass
class GemvCase:
    """One GEMV problem: weight bytes, fp32 activations and the format."""
    fmt: str
    m: int
    n: int
    k: int
    w: np.ndarray
    x: np.ndarray
    meta: dict = field(default_factory=dict)


def gemv_case(fmt: str, m: int, n: int, k: int, seed: int = 0, stream: int = 0,
              weights: np.ndarray | None = None) -> GemvCase:
    """Weights and activations of one GEMV problem.  The weights depend only on
    (fmt, n, k, seed, stream), not on m; pass `weights` to reuse them."""
    if fmt not in ("q4_0", "q8_0"):
        raise ValueError(fmt)
    if weights is not None:
        w = weights
    elif fmt == "q4_0":
        w = q4_0_weights(n, k, seed, 2 * stream)
    else:
        w = q8_0_weights(n, k, seed, 2 * stream)
    x = activations_f32(m, k, seed, 2 * stream + 1 + (1 << 20))
    return GemvCase(fmt, m, n, k, w, x)


def gemm_case(m: int, n: int, k: int, seed: int = 0, stream: int = 0):
    """(Q4_0 weight bytes [n, k/32*18], bf16 bits [m, k])."""
    w = q4_0_weights(n, k, seed, 2 * stream)
    x = activations_bf16(m, k, seed, 2 * stream + 1 + (1 << 21))
    return w, x
