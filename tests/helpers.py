"""Shared test helpers: tolerance checks and device placement.

Tolerances (per output, against the binary64 oracle):
  GEMV (fp32 arithmetic):            |y - y_ref| <= 1e-4 * sum|w*x| + 1e-6
  GEMM (bf16 weights, fp32 sums):    |y - y_ref| <= 2e-3 * sum|w*x| + 1e-6
"""
import numpy as np

GEMV_REL = 1e-4
GEMM_REL = 2e-3
ABS = 1e-6


def assert_within(y, y_ref, bound, rel, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    lim = rel * bound + ABS
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside tolerance; first "
            + ", ".join(f"{tuple(i)}: y={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} "
                        f"bound={bound[tuple(i)]!r}" for i in idx))
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


def to_dev(a, torch, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bf16_tensor(bits, torch, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16).to(device)
