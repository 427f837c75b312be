"""fp64 CPU oracle for the FP8 attention forward: block-wise quantisation with
incoherent processing.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA path.

Source: [P2] zzszmyf.github.io notes, "FlashAttention 原理是什么？为什么又省显存又快",
§10 item ③ (FP8 tensor cores with block-level quantisation plus incoherent
processing, a rotation or permutation that spreads outliers, to keep the
precision loss small) and §12.2 (a scale per block is steadier than one per
tensor; incoherent processing lowers the FP8 attention error further).  The
pages give no formulas; the readings taken:

* FP8 format: OCP E4M3 ("e4m3fn"): 1 sign, 4 exponent bits with bias 7, 3
  mantissa bits, subnormals, no infinities, largest finite 448.  Rounding is
  to nearest, ties to even; values beyond 448 saturate to +-448.
* Incoherent processing: q' = (q * sigma) H / sqrt(d) and k' = (k * sigma) H /
  sqrt(d) for each row, H the d x d Sylvester Hadamard matrix and sigma a
  vector of random signs (an input).  H H^T = d I and sigma^2 = 1, so
  q' . k' = q . k: the scores are unchanged in exact arithmetic, while a
  large coordinate of q or k is spread over all d coordinates.  V is not
  rotated (it does not meet K in a dot product).
* Blocks: one scale per 128-row tile of one (batch, head) of Q', K' and V,
  s = max|x| / 448 over the tile (s = 1 for an all-zero tile); the stored
  value is e4m3(x / s), its meaning s * e4m3(x / s).
* Attention is then the exact attention of the dequantised Q', K', V (computed
  here in fp64 by the plain definition, ``naive_attention``).  The kernel also
  rounds P to e4m3 before its product with V; that rounding is not part of this
  reference, and ``fp8_attention(..., quantize_p=True)`` applies one such
  rounding (at the final row max) to measure how large its effect is.
"""
from __future__ import annotations

import numpy as np

from .attention import naive_attention

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9
BLOCK_ROWS = 128


def e4m3_values() -> np.ndarray:
    """Every finite non-negative E4M3 value, ascending, from the bit layout."""
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue  # the NaN code
            if e == 0:
                vals.append(m * E4M3_SUBNORMAL_STEP)  # subnormal: m/8 * 2^-6
            else:
                vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_POS = e4m3_values()


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value (ties to the even code), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    idx = np.searchsorted(_POS, a)  # _POS[idx - 1] < a <= _POS[idx]
    idx = np.clip(idx, 1, len(_POS) - 1)
    lo, hi = _POS[idx - 1], _POS[idx]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (idx % 2 == 0))  # code idx is even
    r = np.where(pick_hi, hi, lo)
    r = np.where(a == 0.0, 0.0, r)
    return np.copysign(r, x)


def hadamard(d: int) -> np.ndarray:
    """The d x d Sylvester Hadamard matrix (d a power of two), entries +-1."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(x, signs) -> np.ndarray:
    """Incoherent processing of each row: (x * signs) H / sqrt(d)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / np.sqrt(d)


def quantize_blocks(x, block_rows: int = BLOCK_ROWS):
    """Per-tile E4M3 quantisation of the rows of x [N, d].

    Returns (codes as their float64 values, scales [ceil(N / block_rows)]); the
    dequantised tensor is codes * scale of the row's tile."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[0]
    n_tiles = (n + block_rows - 1) // block_rows
    codes = np.empty_like(x)
    scales = np.empty(n_tiles)
    for t in range(n_tiles):
        blk = x[t * block_rows:(t + 1) * block_rows]
        amax = float(np.abs(blk).max()) if blk.size else 0.0
        s = amax / E4M3_MAX if amax > 0.0 else 1.0
        scales[t] = s
        codes[t * block_rows:(t + 1) * block_rows] = e4m3_round(blk / s)
    return codes, scales


def dequantize_blocks(codes, scales, block_rows: int = BLOCK_ROWS) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.float64)
    row_scale = np.repeat(np.asarray(scales, dtype=np.float64), block_rows)[: codes.shape[0]]
    return codes * row_scale[:, None]


def fp8_inputs(q, k, v, signs, rotate_qk: bool = True, block_rows: int = BLOCK_ROWS):
    """The dequantised Q', K', V one (batch, head) slice is attended with."""
    qr = rotate(q, signs) if rotate_qk else np.asarray(q, dtype=np.float64)
    kr = rotate(k, signs) if rotate_qk else np.asarray(k, dtype=np.float64)
    out = []
    for x in (qr, kr, np.asarray(v, dtype=np.float64)):
        codes, scales = quantize_blocks(x, block_rows)
        out.append(dequantize_blocks(codes, scales, block_rows))
    return tuple(out)


def fp8_attention(q, k, v, scale: float, causal: bool, signs, rotate_qk: bool = True,
                  rows=None, quantize_p: bool = False, p_gain: float = 64.0,
                  block_rows: int = BLOCK_ROWS):
    """FP8 attention of one (batch, head) slice: exact attention of the block-quantised,
    rotated inputs.  Returns (O, LSE) in fp64.

    quantize_p=True also rounds each probability to E4M3 before the product with V:
    p_ij = exp(scale s_ij - m_i) (m_i the row max), stored as e4m3(p_ij * p_gain * r_j) and
    used as that value / (p_gain * r_j), r_j = sv_j / max_t sv_t the ratio of key j's V tile
    scale to the largest; l and LSE stay exact.  It is one plausible placement of the
    rounding, for sizing the kernel's tolerance, not a bit-level model of the kernel."""
    qd, kd, vd = fp8_inputs(q, k, v, signs, rotate_qk, block_rows)
    if not quantize_p:
        return naive_attention(qd, kd, vd, scale, causal, rows=rows)
    n, nk = qd.shape[0], kd.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    s = scale * (qd[rows] @ kd.T)
    if causal:
        s = np.where(np.arange(nk)[None, :] > rows[:, None], -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1)
    _, sv = quantize_blocks(np.asarray(v, dtype=np.float64), block_rows)
    ratio = np.repeat(sv / sv.max(), block_rows)[:nk]
    pq = e4m3_round(p * p_gain * ratio[None, :]) / (p_gain * ratio[None, :])
    o = (pq @ vd) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return o, lse
