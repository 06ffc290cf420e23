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


# GeGLU h = gelu(g) * u: the GEMV error of g (scaled by max|gelu'| = 1.1290
# of the tanh form) and of u, plus the fp32 evaluation of the GELU, whose
# argument a ~ g^3 carries a relative error of a few ulp (relative error of
# gelu(g) about 4e-7 * |a| <= 1e-5 * (1 + g^2)).
GELU_SLOPE_MAX = 1.13


def geglu_limit(h_ref, g, u, bound_g, bound_u, rel=GEMV_REL, out_rel=0.0):
    """rel: the products' bound (GEMV 1e-4, GEMM 2e-3); out_rel: rounding of
    the stored h (2^-8 covers bf16 round-to-nearest with margin)."""
    e_g = rel * bound_g + ABS
    e_u = rel * bound_u + ABS
    gelu_g = np.divide(h_ref, u, out=np.zeros_like(h_ref), where=u != 0)
    return (GELU_SLOPE_MAX * np.abs(u) * e_g + np.abs(gelu_g) * e_u
            + (out_rel + 1e-5 * (1.0 + g * g)) * np.abs(h_ref) + ABS)


def assert_geglu_within(h, h_ref, g, u, bound_g, bound_u, what="", rel=GEMV_REL, out_rel=0.0):
    h = np.asarray(h, dtype=np.float64)
    err = np.abs(h - h_ref)
    lim = geglu_limit(h_ref, g, u, bound_g, bound_u, rel, out_rel)
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside tolerance; first "
            + ", ".join(f"{tuple(i)}: h={h[tuple(i)]!r} ref={h_ref[tuple(i)]!r} "
                        f"g={g[tuple(i)]!r} u={u[tuple(i)]!r}" for i in idx))
