"""Parity bar between the CUDA path and the fp64 oracle.

An element passes iff |x_gpu - x_ref| <= tol + ulp/2, where ulp is the unit
in the last place of the output type (fp16: 10 fraction bits, bf16: 7) at
max(|x_ref|, |x_gpu|): the fp32 result is rounded once to the 16-bit output,
which alone costs up to half an ulp (for bf16 |x| in [4, 8) that is 0.0156,
more than the 1e-2 output tolerance). tol is 1e-2 for O, 2e-2 for dQ, dK,
dV; LSE is fp32 and gets the raw 1e-3. Infinities must match exactly.
"""
import numpy as np
import torch

TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD = 2e-2

_FRAC_BITS = {torch.float16: 10, torch.bfloat16: 7, torch.float32: 23}


def half_ulp(x: np.ndarray, dtype) -> np.ndarray:
    bits = _FRAC_BITS[dtype]
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    if dtype == torch.float16:
        e = np.maximum(e, -14.0)
    elif dtype == torch.bfloat16:
        e = np.maximum(e, -126.0)
    return 0.5 * np.exp2(e - bits)


def to_np(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def check(name, got, ref, tol, dtype, report=None):
    """Assert element-wise parity; returns (max raw |diff|, max |ref|)."""
    g = to_np(got)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    fin = np.isfinite(r)
    bad_inf = (not np.array_equal(np.isfinite(g), fin)) or (not np.array_equal(g[~fin], r[~fin]))
    assert not bad_inf, f"{name}: non-finite entries differ (gpu non-finite: {np.sum(~np.isfinite(g))}, ref: {np.sum(~fin)})"
    diff = np.abs(g[fin] - r[fin])
    allowed = tol + (half_ulp(np.maximum(np.abs(g[fin]), np.abs(r[fin])), dtype)
                     if dtype != torch.float32 else 0.0)
    worst = float(np.max(diff, initial=0.0))
    over = diff > allowed
    if report is not None:
        report[name] = {"max_abs_diff": worst, "max_abs_ref": float(np.max(np.abs(r[fin]), initial=0.0))}
    if np.any(over):
        idx = np.argwhere(fin)[np.argmax(diff - allowed)]
        raise AssertionError(
            f"{name}: {int(over.sum())}/{over.size} elements out of tolerance; worst at {tuple(idx)}: "
            f"gpu {g[tuple(idx)]!r} ref {r[tuple(idx)]!r} (tol {tol} + ulp/2)")
    return worst, float(np.max(np.abs(r[fin]), initial=0.0))


# Unit roundoff (half an ulp at 1) of the 16-bit types: round to nearest
# even moves a normal value by at most this fraction of itself.
UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def check_residual(name, o, o_res, o_ref, o_abs_ref, dtype, slack=2e-4):
    """O + o_res is the fp32 result of the P V product before its rounding to
    16 bits. The forward rounds each probability p (<= 1) to the input type
    before that product, which moves p by at most u p (u the unit roundoff;
    fp16 values below 2^-14 by at most 2^-25), so every element obeys
    |O + o_res - O_exact| <= u * (attention applied to |V|) + slack, the slack
    covering fp32 accumulation, ex2.approx and the rounding of o_res itself.
    o_abs_ref is the oracle's attention on |V| for the same scores."""
    got = to_np(o) + to_np(o_res)
    r = np.asarray(o_ref, dtype=np.float64)
    bound = UNIT_ROUNDOFF[dtype] * np.asarray(o_abs_ref, dtype=np.float64) + slack
    diff = np.abs(got - r)
    over = diff > bound
    if np.any(over):
        idx = np.unravel_index(np.argmax(diff - bound), diff.shape)
        raise AssertionError(f"{name}: {int(over.sum())}/{over.size} elements of O + o_res beyond "
                             f"u |O|_abs + {slack}; worst at {idx}: {got[idx]!r} vs {r[idx]!r} "
                             f"(bound {bound[idx]!r})")
    return float(diff.max(initial=0.0))
