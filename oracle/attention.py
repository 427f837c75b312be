"""Plain fp64 CPU oracle for exact attention forward: O and the per-row logsumexp.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA path.

Sources (three web pages on FlashAttention; cited by page and section):

* [P1] aiqz.cc, "flash-attention-io-optimization" article -- sections
  "标准注意力瓶颈" (standard three-step attention), "在线Softmax算法" (the
  unnormalised online update: m_new, r, l_new, O~_new, O = O~/l) and
  "Python 演示" (a blocked NumPy self-check with no scale).
* [P2] zzszmyf.github.io notes, "FlashAttention 原理是什么？为什么又省显存又快" --
  §2 (S = QK^T, P = softmax(S), O = PV), §5 (online softmax in the normalised
  FA1 form), §5.1 (why it is exact), §7.1 (Algorithm 1), §8 (the hand-worked
  example) and §14 exercises 1, 2 and 6.
* [P3] cf-1.com news 5932506 (FlashAttention / roofline blog) -- §3.1 (safe
  softmax: m, l, exp(x - m)/l), §3.2 (running max / running sum merge), §4.3
  (rescale with the running max, not the tile max).

Readings taken where the pages are silent:

* scale: every routine applies ``scale`` to S = Q K^T before the softmax; the
  [P1] demo is the special case scale = 1.
* LSE: natural log, LSE_i = m_i + ln(l_i) = ln sum_j exp(scale * q_i . k_j)
  over the unmasked j.
* causal: key j is masked for query i when its position k_offset + j exceeds the query's
  position q_offset + i.  With q_offset = k_offset = 0 this is the square, top-left
  aligned mask (j > i); decoding appends the Nq new queries after the Nk - Nq cached
  keys, i.e. q_offset = Nk - Nq (bottom-right alignment).
* a query row that sees no key at all (possible only with offsets) has O = 0 and
  LSE = -inf: the empty sum.
* m starts at -inf; the one undefined case, (-inf) - (-inf) when a row has seen
  no unmasked key yet, is guarded explicitly (r = 0, block weights 0).

Every function here works on one (batch, head) slice: q is [Nq, d], k and v are
[N, d], all float64 (bf16 inputs convert to float64 exactly).  ``rows`` selects
which query rows of the slice to compute; rows are independent by definition,
so computing a subset is exact.

Parity pins (see ``tests/test_oracle.py``): the [P2] §8 worked example and its
§14 re-split, brute force on tiny inputs, scipy's softmax / logsumexp, closed
forms (causal row 0, constant scores), and invariants (P rows sum to 1, blocked
== naive for every split, convex hull, shift and permutation invariance, +-30
score rows).  No function here is unpinned.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

NEG_INF = -np.inf


def _query_positions(n_queries: int, rows) -> np.ndarray:
    if rows is None:
        return np.arange(n_queries, dtype=np.int64)
    return np.asarray(rows, dtype=np.int64)


def _finish(acc_or_e_v, l, m):
    """O = acc / l and LSE = m + ln l, with the empty-row convention (l = 0):
    O = 0 and LSE = -inf."""
    empty = ~(l > 0)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(empty[:, None], 0.0, acc_or_e_v / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, -np.inf, m + np.log(np.where(empty, 1.0, l)))
    return out.astype(acc_or_e_v.dtype), lse.astype(acc_or_e_v.dtype)


def _scores(q_rows: np.ndarray, k: np.ndarray, scale: float, causal: bool,
            q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """S = scale * Q K^T for the given query rows and key columns, causal mask
    applied as -inf ([P2] §2, the first of the three steps; mask: j > i)."""
    s = scale * (q_rows @ k.T)
    if causal:
        s = np.where(k_pos[None, :] > q_pos[:, None], NEG_INF, s)
    return s


def naive_attention(q, k, v, scale: float, causal: bool = False, rows=None,
                    row_chunk: int = 256, dtype=np.float64, q_offset: int = 0,
                    k_offset: int = 0):
    """The plain definition, row chunk by row chunk.

    [P2] §2 / [P3] §2.1: S = Q K^T, P = softmax(S) by rows, O = P V, with the
    safe softmax of [P3] §3.1 (m = row max, l = sum exp(s - m), P = exp(s-m)/l).
    LSE = m + ln l.  Row chunking is exact: rows are independent.

    ``q_offset`` / ``k_offset`` are the sequence positions of q's row 0 and k's row 0
    for the causal mask.  Returns (O [len(rows), d], LSE [len(rows)]) in ``dtype``.
    """
    q = np.asarray(q, dtype=dtype)
    k = np.asarray(k, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    q_rows = _query_positions(q.shape[0], rows)
    k_pos = k_offset + np.arange(k.shape[0], dtype=np.int64)
    out = np.empty((q_rows.shape[0], v.shape[1]), dtype=dtype)
    lse = np.empty((q_rows.shape[0],), dtype=dtype)
    for c0 in range(0, q_rows.shape[0], row_chunk):
        idx = q_rows[c0:c0 + row_chunk]
        s = _scores(q[idx], k, dtype(scale), causal, q_offset + idx, k_pos)
        m = s.max(axis=1)
        seen = m > NEG_INF
        with np.errstate(invalid="ignore"):
            e = np.where(seen[:, None], np.exp(s - m[:, None]), 0.0).astype(dtype)
        l = e.sum(axis=1)
        out[c0:c0 + row_chunk], lse[c0:c0 + row_chunk] = _finish(e @ v, l, m)
    return out, lse


def attention_probabilities(q, k, scale: float, causal: bool = False):
    """P = softmax(scale * Q K^T) in full (small N only) -- [P2] §2 step two."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    pos_q = np.arange(q.shape[0], dtype=np.int64)
    pos_k = np.arange(k.shape[0], dtype=np.int64)
    s = _scores(q, k, scale, causal, pos_q, pos_k)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    return e / e.sum(axis=1)[:, None]


def _block_bounds(n_keys: int, block_sizes: Sequence[int] | int) -> list:
    if isinstance(block_sizes, (int, np.integer)):
        size = int(block_sizes)
        if size <= 0:
            raise ValueError("block size must be positive")
        block_sizes = [min(size, n_keys - a) for a in range(0, n_keys, size)]
    bounds, a = [], 0
    for size in block_sizes:
        if size <= 0:
            raise ValueError("block sizes must be positive")
        bounds.append((a, a + int(size)))
        a += int(size)
    if a != n_keys:
        raise ValueError(f"block sizes sum to {a}, expected {n_keys}")
    return bounds


def blocked_online_attention(q, k, v, scale: float, causal: bool = False,
                             block_sizes: Sequence[int] | int = 128, rows=None,
                             dtype=np.float64, trace: list | None = None,
                             q_offset: int = 0, k_offset: int = 0):
    """Online softmax over K/V blocks, unnormalised accumulator form.

    [P1] "在线Softmax算法" and [P3] §3.2: for each block,
        m_new = max(m, m_ij),  r = e^(m - m_new),
        l_new = r l + sum_j e^(s_ij - m_new),
        O~_new = r O~ + sum_j e^(s_ij - m_new) v_j,
    and after the last block O = O~ / l.  m starts at -inf, l and O~ at 0.
    ``block_sizes`` is an int (equal blocks, last one short) or an explicit
    list of block lengths summing to N.  LSE = m + ln l.

    If ``trace`` is a list, (m, l, O~ / l) after each block is appended to it.
    """
    q = np.asarray(q, dtype=dtype)
    k = np.asarray(k, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    q_rows = _query_positions(q.shape[0], rows)
    q_pos = q_offset + q_rows
    qr = q[q_rows]
    m = np.full(q_rows.shape[0], NEG_INF, dtype=dtype)
    l = np.zeros(q_rows.shape[0], dtype=dtype)
    acc = np.zeros((q_rows.shape[0], v.shape[1]), dtype=dtype)
    for a, b in _block_bounds(k.shape[0], block_sizes):
        k_pos = k_offset + np.arange(a, b, dtype=np.int64)
        s_ij = _scores(qr, k[a:b], dtype(scale), causal, q_pos, k_pos)
        m_ij = s_ij.max(axis=1)
        m_new = np.maximum(m, m_ij)
        seen = m_new > NEG_INF          # row has met an unmasked key
        with np.errstate(invalid="ignore"):
            r = np.where(seen, np.exp(m - m_new), 0.0).astype(dtype)
            p_ij = np.where(seen[:, None], np.exp(s_ij - m_new[:, None]), 0.0).astype(dtype)
        l = r * l + p_ij.sum(axis=1)
        acc = r[:, None] * acc + p_ij @ v[a:b]
        m = m_new
        if trace is not None:
            with np.errstate(invalid="ignore", divide="ignore"):
                trace.append((m.copy(), l.copy(), acc / l[:, None]))
    return _finish(acc, l, m)


def blocked_normalised_attention(q, k, v, scale: float, causal: bool = False,
                                 block_sizes: Sequence[int] | int = 128, rows=None,
                                 trace: list | None = None):
    """Online softmax in the normalised form of FA1 ([P2] §5, §7.1 Algorithm 1).

    Per block: m~ = rowmax(S_ij), P~ = exp(S_ij - m~), l~ = rowsum(P~);
        m_new = max(m, m~),
        l_new = e^(m - m_new) l + e^(m~ - m_new) l~,
        O_new = (e^(m - m_new) l O + e^(m~ - m_new) P~ V_j) / l_new.
    O stays normalised after every block.  A block that is fully masked for a
    row (m~ = -inf) contributes nothing to that row.

    If ``trace`` is a list, (m, l, O, m~, P~, l~) after each block is appended.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    q_pos = _query_positions(q.shape[0], rows)
    qr = q[q_pos]
    m = np.full(q_pos.shape[0], NEG_INF)
    ell = np.zeros(q_pos.shape[0])
    out = np.zeros((q_pos.shape[0], v.shape[1]))
    for a, b in _block_bounds(k.shape[0], block_sizes):
        k_pos = np.arange(a, b, dtype=np.int64)
        s_ij = _scores(qr, k[a:b], scale, causal, q_pos, k_pos)
        m_t = s_ij.max(axis=1)
        live = m_t > NEG_INF            # block holds an unmasked key for the row
        with np.errstate(invalid="ignore"):
            p_t = np.where(live[:, None], np.exp(s_ij - m_t[:, None]), 0.0)
        l_t = p_t.sum(axis=1)
        m_new = np.maximum(m, m_t)
        seen = m_new > NEG_INF
        with np.errstate(invalid="ignore"):
            a_old = np.where(seen & (m > NEG_INF), np.exp(m - m_new), 0.0)
            a_new = np.where(seen & live, np.exp(m_t - m_new), 0.0)
        l_new = a_old * ell + a_new * l_t
        with np.errstate(invalid="ignore", divide="ignore"):
            out = np.where(seen[:, None],
                           ((a_old * ell)[:, None] * out + a_new[:, None] * (p_t @ v[a:b]))
                           / l_new[:, None],
                           0.0)
        m, ell = m_new, l_new
        if trace is not None:
            trace.append((m.copy(), ell.copy(), out.copy(), m_t.copy(), p_t.copy(), l_t.copy()))
    lse = m + np.log(ell)
    return out, lse


def brute_force_attention(q, k, v, scale: float, causal: bool = False, q_offset: int = 0,
                          k_offset: int = 0):
    """A third, scalar implementation for tiny inputs (N <= 16): explicit loops
    over i, j and the head dimension with math.exp, straight from the
    definition softmax(s)_j = exp(s_j - m) / sum_k exp(s_k - m) ([P3] §3.1)."""
    q = [[float(x) for x in row] for row in np.asarray(q, dtype=np.float64)]
    k = [[float(x) for x in row] for row in np.asarray(k, dtype=np.float64)]
    v = [[float(x) for x in row] for row in np.asarray(v, dtype=np.float64)]
    n_q, n_k, d_v = len(q), len(k), len(v[0])
    out = [[0.0] * d_v for _ in range(n_q)]
    lse = [0.0] * n_q
    for i in range(n_q):
        allowed = [j for j in range(n_k) if not (causal and k_offset + j > q_offset + i)]
        if not allowed:  # empty sum: O = 0, LSE = -inf
            lse[i] = -math.inf
            continue
        s = {}
        for j in allowed:
            dot = 0.0
            for c in range(len(q[i])):
                dot += q[i][c] * k[j][c]
            s[j] = scale * dot
        m = max(s.values())
        denom = 0.0
        for j in allowed:
            denom += math.exp(s[j] - m)
        for c in range(d_v):
            num = 0.0
            for j in allowed:
                num += math.exp(s[j] - m) * v[j][c]
            out[i][c] = num / denom
        lse[i] = m + math.log(denom)
    return np.array(out), np.array(lse)


def split_kv_attention(q, k, v, scale: float, causal: bool = False,
                       split_sizes: Sequence[int] | int = 128, rows=None,
                       q_offset: int = 0):
    """Split-KV attention as in FlashDecoding ([P2] §12.1): each split of the keys
    gives a partial result (O_s, LSE_s) computed on its own (``naive_attention`` on the
    split, with the split's key positions), and the partials merge exactly:
        LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
    Splits with no visible key (LSE_s = -inf) contribute nothing.
    """
    parts = []
    for a, b in _block_bounds(np.asarray(k).shape[0], split_sizes):
        parts.append(naive_attention(q, np.asarray(k)[a:b], np.asarray(v)[a:b], scale, causal,
                                     rows=rows, q_offset=q_offset, k_offset=a))
    lse_s = np.stack([p[1] for p in parts])            # [S, rows]
    o_s = np.stack([p[0] for p in parts])              # [S, rows, d]
    top = lse_s.max(axis=0)
    seen = top > NEG_INF
    with np.errstate(invalid="ignore"):
        w = np.where(seen[None, :], np.exp(lse_s - np.where(seen, top, 0.0)[None, :]), 0.0)
    total = w.sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(seen[:, None], (w[:, :, None] * o_s).sum(axis=0) / np.where(seen, total, 1.0)[:, None], 0.0)
        lse = np.where(seen, top + np.log(np.where(seen, total, 1.0)), NEG_INF)
    return out, lse


def attention_backward(q, k, v, do, scale: float, causal: bool = False, q_offset: int = 0):
    """Gradients of O = softmax(scale Q K^T) V for an upstream gradient dO.

    The recompute scheme of [P2] §6 (and [P1] 工程实现细节) keeps only the per-row
    statistics of the forward; the gradients follow from the chain rule through
    O = P V and P = softmax(S), S = scale Q K^T:
        D_i   = sum_c dO_ic O_ic           (= sum_j P_ij dP_ij)
        dV    = P^T dO
        dP    = dO V^T
        dS    = P * (dP - D)               (softmax Jacobian, row by row)
        dQ    = scale dS K,    dK = scale dS^T Q.
    Masked entries have P = 0, so they contribute nothing.  Rows that see no key
    (only with offsets) have P = 0 and zero gradients.  Returns (dQ, dK, dV, D) in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    q_pos = q_offset + np.arange(q.shape[0], dtype=np.int64)
    k_pos = np.arange(k.shape[0], dtype=np.int64)
    s = _scores(q, k, scale, causal, q_pos, k_pos)
    m = s.max(axis=1)
    seen = m > NEG_INF
    with np.errstate(invalid="ignore"):
        e = np.where(seen[:, None], np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    p = e / np.where(seen, l, 1.0)[:, None]
    o = p @ v
    d_row = (do * o).sum(axis=1)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - d_row[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, d_row


def naive_attention_bhnd(q, k, v, scale: float, causal: bool = False,
                         slices: Iterable | None = None, rows=None):
    """Apply ``naive_attention`` to each (b, h) slice of [B, H, N, d] arrays.

    ``slices`` lists the (b, h) pairs to compute (default: all).  Returns a
    dict {(b, h): (O, LSE)} -- every slice is an independent problem.
    """
    bsz, heads = q.shape[0], q.shape[1]
    if slices is None:
        slices = [(b, h) for b in range(bsz) for h in range(heads)]
    return {(b, h): naive_attention(q[b, h], k[b, h], v[b, h], scale, causal, rows=rows)
            for (b, h) in slices}
