"""Parity helpers shared by the GPU tests and bench.py (no attention arithmetic).

Tolerances (bf16 in, fp32 accumulate, bf16 O out, fp32 LSE):
  * max |dO| <= 1e-2, raw, on every element whose fp64 value bf16 can represent to
    within 1e-2: every |O_ref| < 4, where half a bf16 ulp is at most 2^-7 = 0.0078.
    For |O_ref| >= 4 half a bf16 ulp is 2^-6 = 0.0156 or more, so no bf16 output can
    promise 1e-2 there; those elements may differ by 1e-2 + half an ulp of O_ref.
  * mean |dO| <= 1e-3, raw, over every element compared.
  * LSE: |dLSE| <= 1e-3 * max(1, |LSE|).
The raw max |dO| over all elements and over the |O_ref| < 4 elements are both
reported.

Backward (bf16 dQ, dK, dV; P and dS rounded to bf16 before their products, fp32
accumulation, D from the forward's bf16 O): errors are measured relative to the
size of the gradient itself, max |d| <= 2e-2 * max |ref| and mean |d| <= 1e-2 *
mean |ref|.  A replay of exactly that rounding in fp64 on the test shapes gives
2.5e-3 to 5.3e-3 on both measures (the upper end with score std 3), so the bounds
leave a factor of about 2 to 4.  D = rowsum(dO * O) is held to the same two
relative bounds (its error comes from the bf16 rounding of O).
"""
from __future__ import annotations

import json
import os

import numpy as np

MAX_ABS_O = 1e-2
MEAN_ABS_O = 1e-3
LSE_REL = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) around |x|."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(ax, 2.0 ** -126))   # ax = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9)


def o_allowance(o_ref: np.ndarray) -> np.ndarray:
    """Per-element bound on |dO|: 1e-2 where half a bf16 ulp of O_ref is below 1e-2
    (|O_ref| < 4), else 1e-2 plus that half ulp."""
    half = bf16_half_ulp(o_ref)
    return np.where(half < MAX_ABS_O, MAX_ABS_O, MAX_ABS_O + half)


def compare(o_gpu, lse_gpu, o_ref, lse_ref) -> dict:
    """Error statistics of one result against the oracle.  Rows the oracle marks
    empty (LSE = -inf, O = 0) must be empty on the GPU too."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    d_o = np.abs(o_gpu - o_ref)
    small = bf16_half_ulp(o_ref) < MAX_ABS_O
    over = d_o - o_allowance(o_ref)
    fin = np.isfinite(lse_ref)
    same_empty = bool(np.array_equal(np.isneginf(lse_gpu), np.isneginf(lse_ref)))
    d_l = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    return {
        "max_abs_o": float(d_o.max()) if d_o.size else 0.0,
        "max_abs_o_below4": float(d_o[small].max()) if small.any() else 0.0,
        "max_abs_o_over_allowance": float(over.max()) if over.size else -MAX_ABS_O,
        "mean_abs_o": float(d_o.mean()) if d_o.size else 0.0,
        "max_rel_lse": float(d_l.max()) if d_l.size else 0.0,
        "finite": bool(np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu[fin]))) and same_empty,
        "count": int(d_o.size),
    }


def merge(stats: list) -> dict:
    """Statistics of several compared parts taken together (means weighted by count)."""
    if not stats:
        raise ValueError("nothing compared")
    return {
        "max_abs_o": max(s["max_abs_o"] for s in stats),
        "max_abs_o_below4": max(s["max_abs_o_below4"] for s in stats),
        "max_abs_o_over_allowance": max(s["max_abs_o_over_allowance"] for s in stats),
        "mean_abs_o": float(np.average([s["mean_abs_o"] for s in stats], weights=[max(s["count"], 1) for s in stats])),
        "max_rel_lse": max(s["max_rel_lse"] for s in stats),
        "finite": all(s["finite"] for s in stats),
        "count": sum(s["count"] for s in stats),
    }


def log_stats(name: str, st: dict, slices, rows_per_slice: int) -> None:
    """Append one JSON line of raw error statistics to the file FA_PARITY_LOG names, if any."""
    path = os.environ.get("FA_PARITY_LOG")
    if path:
        with open(path, "a", encoding="utf-8") as f:
            f.write(json.dumps({"workload": name, "slices": len(slices), "rows_per_slice": rows_per_slice,
                                **st}) + "\n")


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
    return (st["finite"] and st["max_abs_o_over_allowance"] <= 0.0
            and st["mean_abs_o"] <= MEAN_ABS_O and st["max_rel_lse"] <= LSE_REL)
