"""Parity helpers shared by the GPU tests and bench.py (no attention arithmetic).

Tolerances (bf16 in, fp32 accumulate, bf16 O out, fp32 LSE):
  * max |dO| <= 1e-2 once the output's own bf16 rounding is set aside: each
    element may differ from the fp64 value by 1e-2 + half a bf16 ulp of that
    value.  (A bf16 O cannot be closer than half an ulp, and for |O| >= 4 half
    an ulp alone exceeds 1e-2.)  The raw max |dO| is reported as well.
  * mean |dO| <= 1e-3, raw.
  * LSE: |dLSE| <= 1e-3 * max(1, |LSE|).

Backward (bf16 dQ, dK, dV; P and dS rounded to bf16 before their products, fp32
accumulation, D from the forward's bf16 O): errors are measured relative to the
size of the gradient itself, max |d| <= 2e-2 * max |ref| and mean |d| <= 1e-2 *
mean |ref|.  A replay of exactly that rounding in fp64 on the test shapes gives
2.5e-3 to 5.3e-3 on both measures (the upper end with score std 3), so the bounds
leave a factor of about 2 to 4.  D = rowsum(dO * O) is held to the same two
relative bounds (its error comes from the bf16 rounding of O).
"""
from __future__ import annotations

import numpy as np

MAX_ABS_O = 1e-2
MEAN_ABS_O = 1e-3
LSE_REL = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) around |x|."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(ax, 2.0 ** -126))   # ax = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9)


def compare(o_gpu, lse_gpu, o_ref, lse_ref) -> dict:
    """Error statistics of one result against the oracle.  Rows the oracle marks
    empty (LSE = -inf, O = 0) must be empty on the GPU too."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    d_o = np.abs(o_gpu - o_ref)
    excess = np.maximum(d_o - bf16_half_ulp(o_ref), 0.0)
    fin = np.isfinite(lse_ref)
    same_empty = bool(np.array_equal(np.isneginf(lse_gpu), np.isneginf(lse_ref)))
    d_l = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    return {
        "max_abs_o": float(d_o.max()) if d_o.size else 0.0,
        "max_abs_o_beyond_output_rounding": float(excess.max()) if excess.size else 0.0,
        "mean_abs_o": float(d_o.mean()) if d_o.size else 0.0,
        "max_rel_lse": float(d_l.max()) if d_l.size else 0.0,
        "finite": bool(np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu[fin]))) and same_empty,
        "count": int(d_o.size),
    }


GRAD_MAX_REL = 2e-2
GRAD_MEAN_REL = 1e-2


def grad_compare(g_gpu, g_ref) -> dict:
    """Gradient error relative to the gradient's own size."""
    g_gpu = np.asarray(g_gpu, dtype=np.float64)
    g_ref = np.asarray(g_ref, dtype=np.float64)
    diff = np.abs(g_gpu - g_ref)
    ref_max = float(np.abs(g_ref).max()) if g_ref.size else 0.0
    ref_mean = float(np.abs(g_ref).mean()) if g_ref.size else 0.0
    return {
        "max_rel": float(diff.max()) / max(ref_max, 1e-30) if diff.size else 0.0,
        "mean_rel": float(diff.mean()) / max(ref_mean, 1e-30) if diff.size else 0.0,
        "finite": bool(np.all(np.isfinite(g_gpu))),
    }


def grad_within_tolerance(st: dict) -> bool:
    return st["finite"] and st["max_rel"] <= GRAD_MAX_REL and st["mean_rel"] <= GRAD_MEAN_REL


def within_tolerance(st: dict) -> bool:
    return (st["finite"] and st["max_abs_o_beyond_output_rounding"] <= MAX_ABS_O
            and st["mean_abs_o"] <= MEAN_ABS_O and st["max_rel_lse"] <= LSE_REL)
