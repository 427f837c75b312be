"""Pins for the CPU oracle: checks against facts fixed by the pages and by the
mathematics, each a function of the oracle module so a mutated copy of the
oracle can be run through the same checks (``test_oracle_mutants.py``).

Each pin raises AssertionError (or any exception) when the oracle is wrong.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "online_softmax_worked_example.json")


def _rng(seed):
    return np.random.default_rng(seed)


def pin_worked_example(mod):
    """Page 'FlashAttention 原理是什么？…' §8 and §14 exercise 2: the printed
    per-block states of the online softmax and the full-softmax weights."""
    g = json.load(open(GOLDEN, encoding="utf-8"))
    tol3, tol4 = g["tolerance"]["three_decimals"], g["tolerance"]["four_decimals"]
    q = np.array([[1.0]])
    k = np.array(g["scores"], dtype=np.float64)[:, None]      # scores = q.k with scale 1
    v = np.array(g["v"], dtype=np.float64)[:, None]
    for key, sizes in (("split_2_1", [2, 1]), ("split_1_2", [1, 2])):
        tr = []
        o, lse = mod.blocked_normalised_attention(q, k, v, 1.0, False, sizes, trace=tr)
        for blk, state in zip(("block1", "block2"), tr):
            m, ell, out, m_t, p_t, l_t = state
            want = g[key][blk]
            assert abs(m[0] - want["m"]) < tol3, (key, blk, "m")
            assert abs(ell[0] - want["l"]) < tol3, (key, blk, "l", ell[0])
            assert abs(out[0, 0] - want["O"]) < tol3, (key, blk, "O", out[0, 0])
            assert abs(m_t[0] - want["m_tilde"]) < tol3, (key, blk, "m~")
            assert abs(l_t[0] - want["l_tilde"]) < tol3, (key, blk, "l~")
            assert np.allclose(p_t[0], want["P_tilde"], atol=tol3), (key, blk, "P~")
        # the unnormalised form passes through the same running m, l and O~/l
        tr2 = []
        mod.blocked_online_attention(q, k, v, 1.0, False, sizes, trace=tr2)
        assert abs(tr2[-1][1][0] - g[key]["block2"]["l"]) < tol3
        assert abs(tr2[-1][2][0, 0] - g[key]["block2"]["O"]) < tol3
    o, lse = mod.naive_attention(q, k, v, 1.0, False)
    assert abs(o[0, 0] - g["full_softmax"]["O"]) < tol4, o[0, 0]
    p = mod.attention_probabilities(q, k, 1.0, False)
    assert np.allclose(p[0], g["full_softmax"]["a"], atol=tol4), p[0]


def pin_worked_example_exact(mod):
    """The same example in exact arithmetic: s = (sqrt2, 1/sqrt2, 1/sqrt2) gives
    a = (1, e^-c, e^-c)/(1 + 2e^-c) with c = 1/sqrt2; LSE = sqrt2 + ln(1 + 2e^-c)."""
    c = 1.0 / math.sqrt(2.0)
    q = np.array([[1.0]])
    k = np.array([[2 * c], [c], [c]])
    v = np.array([[1.0], [0.0], [1.0]])
    den = 1.0 + 2.0 * math.exp(-c)
    want_o = (1.0 + math.exp(-c)) / den
    want_lse = 2 * c + math.log(den)
    for fn in (lambda: mod.naive_attention(q, k, v, 1.0),
               lambda: mod.blocked_online_attention(q, k, v, 1.0, False, [2, 1]),
               lambda: mod.blocked_online_attention(q, k, v, 1.0, False, [1, 2]),
               lambda: mod.blocked_normalised_attention(q, k, v, 1.0, False, [1, 1, 1])):
        o, lse = fn()
        assert abs(o[0, 0] - want_o) < 1e-14 and abs(lse[0] - want_lse) < 1e-14


def pin_brute_force(mod):
    """Tiny inputs: the vectorised routines equal the scalar triple loop."""
    rng = _rng(1)
    for n, d, causal, scale in ((1, 3, False, 1.0), (4, 3, False, 1.0), (5, 4, True, 0.5),
                                (7, 2, True, 1.3), (8, 5, False, 0.35)):
        q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
        o_b, l_b = mod.brute_force_attention(q, k, v, scale, causal)
        for o, l in (mod.naive_attention(q, k, v, scale, causal, row_chunk=3),
                     mod.blocked_online_attention(q, k, v, scale, causal, 2),
                     mod.blocked_normalised_attention(q, k, v, scale, causal, 3)):
            assert np.max(np.abs(o - o_b)) < 1e-12 and np.max(np.abs(l - l_b)) < 1e-12


def pin_brute_force_by_hand(mod):
    """A 2x2 case worked by hand: q=(1,0),(0,1); k=(1,0),(0,2); v=(1,2),(3,4);
    scale 1.  Row 0 scores (1, 0), row 1 scores (0, 2)."""
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    k = np.array([[1.0, 0.0], [0.0, 2.0]])
    v = np.array([[1.0, 2.0], [3.0, 4.0]])
    w0 = np.array([math.e, 1.0]) / (math.e + 1.0)
    w1 = np.array([1.0, math.e ** 2]) / (1.0 + math.e ** 2)
    want = np.stack([w0 @ v, w1 @ v])
    want_lse = np.array([math.log(math.e + 1.0), math.log(1.0 + math.e ** 2)])
    o, lse = mod.brute_force_attention(q, k, v, 1.0, False)
    assert np.allclose(o, want, atol=1e-14) and np.allclose(lse, want_lse, atol=1e-14)
    o, lse = mod.naive_attention(q, k, v, 1.0, False)
    assert np.allclose(o, want, atol=1e-14) and np.allclose(lse, want_lse, atol=1e-14)
    # causal: row 0 sees key 0 only
    o, lse = mod.naive_attention(q, k, v, 1.0, True)
    assert np.allclose(o[0], v[0]) and abs(lse[0] - 1.0) < 1e-14
    assert np.allclose(o[1], want[1], atol=1e-14)


def pin_scipy(mod):
    """Non-causal rows against scipy.special.softmax / logsumexp (a library
    routine the oracle does not call)."""
    rng = _rng(2)
    n, d = 96, 16
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    scale = 1.0 / math.sqrt(d)
    s = scale * (q @ k.T)
    want_o = scipy.special.softmax(s, axis=1) @ v
    want_lse = scipy.special.logsumexp(s, axis=1)
    o, lse = mod.naive_attention(q, k, v, scale, False, row_chunk=40)
    assert np.max(np.abs(o - want_o)) < 1e-13 and np.max(np.abs(lse - want_lse)) < 1e-12
    # causal via scipy on the lower-triangular prefix of each row
    o, lse = mod.naive_attention(q, k, v, scale, True)
    for i in (0, 1, 17, n - 1):
        w = scipy.special.softmax(s[i, :i + 1])
        assert np.max(np.abs(o[i] - w @ v[:i + 1])) < 1e-13
        assert abs(lse[i] - scipy.special.logsumexp(s[i, :i + 1])) < 1e-12


def pin_probabilities(mod):
    """Rows of P sum to 1 and are non-negative; causal P is lower-triangular."""
    rng = _rng(3)
    q, k = rng.standard_normal((64, 8)), rng.standard_normal((64, 8))
    for causal in (False, True):
        p = mod.attention_probabilities(q, k, 0.7, causal)
        assert np.all(p >= 0) and np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-12
        if causal:
            assert np.all(np.triu(p, 1) == 0.0)


def pin_blocked_equals_naive(mod):
    """Blocked online softmax equals the full softmax for every split (the
    induction of the page's §14 exercise 1), in both the unnormalised and the
    normalised form, with and without the causal mask."""
    rng = _rng(4)
    n, d = 160, 8
    q, k, v = (rng.standard_normal((n, d)) * 2.0 for _ in range(3))
    splits = [1, 2, 8, 32, 128, 160, [100, 60], [1, 159], [159, 1],
              list(rng.integers(1, 20, 200).cumsum())]
    for causal in (False, True):
        o_ref, l_ref = mod.naive_attention(q, k, v, 0.4, causal)
        for sp in splits:
            if isinstance(sp, list) and len(sp) > 3:      # random split points
                cuts = sorted(set(int(c) for c in sp if 0 < c < n))
                bounds = [0] + cuts + [n]
                sp = [b - a for a, b in zip(bounds[:-1], bounds[1:])]
            for fn in (mod.blocked_online_attention, mod.blocked_normalised_attention):
                o, l = fn(q, k, v, 0.4, causal, sp)
                assert np.max(np.abs(o - o_ref)) < 1e-12, (fn.__name__, sp, causal)
                assert np.max(np.abs(l - l_ref)) < 1e-12, (fn.__name__, sp, causal)


def pin_fp32_blocks(mod):
    """The page's exercise 6: in float32 the blocked and full results agree to
    about 1e-7 for block sizes 2, 8, 32, 128."""
    rng = _rng(5)
    q, k, v = (rng.standard_normal((256, 32)).astype(np.float32) for _ in range(3))
    o_ref, _ = mod.naive_attention(q, k, v, 1 / math.sqrt(32), False, dtype=np.float32)
    for bs in (2, 8, 32, 128):
        o, _ = mod.blocked_online_attention(q, k, v, 1 / math.sqrt(32), False, bs, dtype=np.float32)
        assert o.dtype == np.float32
        assert np.max(np.abs(o - o_ref)) < 2e-6, bs


def pin_closed_forms(mod):
    """Causal row 0 equals V[0] with LSE = scale q0.k0; constant scores give the
    mean of the visible V rows and LSE = c + ln(count)."""
    rng = _rng(6)
    n, d = 40, 6
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    o, lse = mod.naive_attention(q, k, v, 0.3, True)
    assert np.max(np.abs(o[0] - v[0])) < 1e-15 and abs(lse[0] - 0.3 * q[0] @ k[0]) < 1e-14
    ob, lb = mod.blocked_online_attention(q, k, v, 0.3, True, 7)
    assert np.max(np.abs(ob[0] - v[0])) < 1e-15 and abs(lb[0] - 0.3 * q[0] @ k[0]) < 1e-14
    # q = 0: all scores 0
    z = np.zeros((n, d))
    o, lse = mod.naive_attention(z, k, v, 0.3, False)
    assert np.max(np.abs(o - v.mean(axis=0))) < 1e-14 and np.max(np.abs(lse - math.log(n))) < 1e-13
    o, lse = mod.naive_attention(z, k, v, 0.3, True)
    for i in range(n):
        assert np.max(np.abs(o[i] - v[:i + 1].mean(axis=0))) < 1e-14
        assert abs(lse[i] - math.log(i + 1)) < 1e-13


def pin_large_scores(mod):
    """Rows of +30 or -30 scores: no overflow, no NaN; O is the mean of the V
    rows and LSE = +-30 + ln(count) (q = c e1, k = e1)."""
    n, d = 64, 4
    rng = _rng(7)
    v = rng.standard_normal((n, d))
    k = np.zeros((n, d)); k[:, 0] = 1.0
    for c in (30.0, -30.0, 300.0, -300.0):
        q = np.zeros((n, d)); q[:, 0] = c
        for fn in (lambda: mod.naive_attention(q, k, v, 1.0, False),
                   lambda: mod.blocked_online_attention(q, k, v, 1.0, False, 16),
                   lambda: mod.blocked_normalised_attention(q, k, v, 1.0, False, 16)):
            o, lse = fn()
            assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
            assert np.max(np.abs(o - v.mean(axis=0))) < 1e-13
            assert np.max(np.abs(lse - (c + math.log(n)))) < 1e-12


def pin_convex_hull(mod):
    """Each O row lies within the per-coordinate range of the visible V rows."""
    rng = _rng(8)
    n, d = 80, 5
    q, k, v = (rng.standard_normal((n, d)) * 3 for _ in range(3))
    for causal in (False, True):
        o, _ = mod.naive_attention(q, k, v, 1.0, causal)
        for i in range(n):
            vis = v[: i + 1] if causal else v
            assert np.all(o[i] >= vis.min(axis=0) - 1e-12) and np.all(o[i] <= vis.max(axis=0) + 1e-12)


def pin_shift_and_permutation(mod):
    """Adding u to every K row leaves O unchanged and shifts LSE_i by
    scale q_i.u; permuting K and V rows together (non-causal) changes nothing;
    softmax is not invariant to permuting K alone (catches a V/K mix-up)."""
    rng = _rng(9)
    n, d, scale = 50, 7, 0.45
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    u = rng.standard_normal(d)
    o, lse = mod.naive_attention(q, k, v, scale, False)
    o2, lse2 = mod.naive_attention(q, k + u, v, scale, False)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse2 - lse - scale * (q @ u))) < 1e-12
    oc, lc = mod.naive_attention(q, k, v, scale, True)
    oc2, lc2 = mod.naive_attention(q, k + u, v, scale, True)
    assert np.max(np.abs(oc - oc2)) < 1e-12 and np.max(np.abs(lc2 - lc - scale * (q @ u))) < 1e-12
    perm = rng.permutation(n)
    o3, lse3 = mod.naive_attention(q, k[perm], v[perm], scale, False)
    assert np.max(np.abs(o - o3)) < 1e-12 and np.max(np.abs(lse - lse3)) < 1e-12
    o4, _ = mod.naive_attention(q, k[perm], v, scale, False)
    assert np.max(np.abs(o - o4)) > 1e-3


def pin_rows_subset(mod):
    """Computing a subset of query rows equals the same rows of the full result."""
    rng = _rng(10)
    q, k, v = (rng.standard_normal((300, 8)) for _ in range(3))
    rows = [0, 5, 128, 255, 299]
    for causal in (False, True):
        o, l = mod.naive_attention(q, k, v, 0.5, causal)
        o2, l2 = mod.naive_attention(q, k, v, 0.5, causal, rows=rows, row_chunk=2)
        o3, l3 = mod.blocked_online_attention(q, k, v, 0.5, causal, 64, rows=rows)
        assert np.max(np.abs(o[rows] - o2)) < 1e-13 and np.max(np.abs(l[rows] - l2)) < 1e-13
        assert np.max(np.abs(o[rows] - o3)) < 1e-12 and np.max(np.abs(l[rows] - l3)) < 1e-12


def pin_offsets_and_empty_rows(mod):
    """Causal masks with sequence offsets against the brute-force loop; rows that
    see no key give O = 0 and LSE = -inf (the empty sum)."""
    rng = _rng(11)
    q, k, v = rng.standard_normal((6, 4)), rng.standard_normal((9, 4)), rng.standard_normal((9, 3))
    for q_off, k_off in ((3, 0), (0, 2), (-2, 0), (5, 5), (8, 0)):
        o_b, l_b = mod.brute_force_attention(q, k, v, 0.7, True, q_offset=q_off, k_offset=k_off)
        for o, l in (mod.naive_attention(q, k, v, 0.7, True, q_offset=q_off, k_offset=k_off, row_chunk=4),
                     mod.blocked_online_attention(q, k, v, 0.7, True, 4, q_offset=q_off, k_offset=k_off)):
            assert np.array_equal(np.isinf(l), np.isinf(l_b))
            fin = np.isfinite(l_b)
            assert np.max(np.abs(o - o_b)) < 1e-12 and np.max(np.abs(l[fin] - l_b[fin])) < 1e-12
        empty = [i for i in range(6) if q_off + i < k_off]
        for i in empty:
            assert np.all(o_b[i] == 0.0) and l_b[i] == -np.inf
    # hand check: q_offset = -1 leaves row 0 empty, row 1 sees key 0 only
    o, l = mod.naive_attention(q[:2], k, v, 1.0, True, q_offset=-1)
    assert np.all(o[0] == 0.0) and l[0] == -np.inf
    assert np.allclose(o[1], v[0]) and abs(l[1] - q[1] @ k[0]) < 1e-14


def pin_decode_alignment(mod):
    """Bottom-right causal decode: one new query at position Nk - 1 sees every key
    (equals non-causal); Nq = Nk with offset 0 is the square mask."""
    rng = _rng(12)
    q, k, v = rng.standard_normal((1, 8)), rng.standard_normal((40, 8)), rng.standard_normal((40, 8))
    o_c, l_c = mod.naive_attention(q, k, v, 0.3, True, q_offset=39)
    o_n, l_n = mod.naive_attention(q, k, v, 0.3, False)
    assert np.max(np.abs(o_c - o_n)) < 1e-14 and np.max(np.abs(l_c - l_n)) < 1e-14
    q4 = rng.standard_normal((4, 8))
    o4, l4 = mod.naive_attention(q4, k, v, 0.3, True, q_offset=36)   # last 4 positions
    for i in range(4):
        oi, li = mod.naive_attention(q4[i:i + 1], k[:37 + i], v[:37 + i], 0.3, False)
        assert np.max(np.abs(o4[i] - oi[0])) < 1e-13 and abs(l4[i] - li[0]) < 1e-13


def pin_split_kv(mod):
    """FlashDecoding merge ([P2] §12.1): split-KV partials merge to the full
    result for every split; the §8 worked example as a 2+1 split gives 0.752."""
    g = json.load(open(GOLDEN, encoding="utf-8"))
    q = np.array([[1.0]])
    k = np.array(g["scores"])[:, None]
    v = np.array(g["v"])[:, None]
    o, lse = mod.split_kv_attention(q, k, v, 1.0, False, [2, 1])
    assert abs(o[0, 0] - g["split_2_1"]["block2"]["O"]) < g["tolerance"]["three_decimals"]
    assert abs(lse[0] - (g["split_2_1"]["block2"]["m"] + math.log(g["split_2_1"]["block2"]["l"]))) < 1e-3
    rng = _rng(13)
    q, k, v = rng.standard_normal((5, 8)), rng.standard_normal((70, 8)), rng.standard_normal((70, 6))
    for causal, q_off in ((False, 0), (True, 65), (True, 30)):
        o_ref, l_ref = mod.naive_attention(q, k, v, 0.4, causal, q_offset=q_off)
        for sp in (1, 7, 16, 70, [3, 60, 7], [69, 1]):
            o, l = mod.split_kv_attention(q, k, v, 0.4, causal, sp, q_offset=q_off)
            fin = np.isfinite(l_ref)
            assert np.array_equal(np.isinf(l), np.isinf(l_ref))
            assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(l[fin] - l_ref[fin])) < 1e-12


def _loss_grad_fd(mod, q, k, v, g, scale, causal, which, idx, h=1e-6):
    """Central difference of L = sum(O * g) with respect to one input element."""
    arrs = {"q": q, "k": k, "v": v}
    a = arrs[which].copy()
    a[idx] += h
    up = dict(arrs, **{which: a})
    o1, _ = mod.naive_attention(up["q"], up["k"], up["v"], scale, causal)
    a[idx] -= 2 * h
    dn = dict(arrs, **{which: a})
    o2, _ = mod.naive_attention(dn["q"], dn["k"], dn["v"], scale, causal)
    return ((o1 - o2) * g).sum() / (2 * h)


def pin_backward_finite_differences(mod):
    """The analytic gradients equal central differences of L = sum(O * dO) in every
    element of Q, K and V (tiny inputs, fp64; error ~1e-9)."""
    rng = _rng(14)
    for n, d, causal, scale in ((5, 3, False, 0.7), (6, 4, True, 1.1)):
        q, k, v, g = (rng.standard_normal((n, d)) for _ in range(4))
        dq, dk, dv, _ = mod.attention_backward(q, k, v, g, scale, causal)
        for which, grad in (("q", dq), ("k", dk), ("v", dv)):
            for idx in np.ndindex(n, d):
                fd = _loss_grad_fd(mod, q, k, v, g, scale, causal, which, idx)
                assert abs(fd - grad[idx]) < 1e-6, (which, idx, fd, grad[idx])


def pin_backward_torch(mod):
    """Against torch.autograd in fp64 on the CPU (a library the oracle does not use)."""
    import torch
    rng = _rng(15)
    n, d, scale = 33, 8, 0.4
    for causal in (False, True):
        arrs = [rng.standard_normal((n, d)) for _ in range(4)]
        q, k, v = (torch.tensor(a, requires_grad=True) for a in arrs[:3])
        g = torch.tensor(arrs[3])
        s = scale * q @ k.T
        if causal:
            s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
        (torch.softmax(s, dim=1) @ v * g).sum().backward()
        dq, dk, dv, _ = mod.attention_backward(*arrs[:3], arrs[3], scale, causal)
        for mine, ref in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
            assert np.max(np.abs(mine - ref.numpy())) < 1e-12


def pin_backward_invariants(mod):
    """Rows of dS sum to zero, so the K gradients sum to zero over keys (scores are
    invariant to adding one vector to every key); uniform attention (q = 0) gives
    dV_j = mean over the queries that see key j of dO_i; D = rowsum(dO * O)."""
    rng = _rng(16)
    n, d = 20, 5
    q, k, v, g = (rng.standard_normal((n, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, drow = mod.attention_backward(q, k, v, g, 0.6, causal)
        assert np.max(np.abs(dk.sum(axis=0))) < 1e-12
        o, _ = mod.naive_attention(q, k, v, 0.6, causal)
        assert np.max(np.abs(drow - (g * o).sum(axis=1))) < 1e-12
    z = np.zeros((n, d))
    dq, dk, dv, _ = mod.attention_backward(z, k, v, g, 0.6, False)
    assert np.max(np.abs(dv - g.mean(axis=0)[None, :])) < 1e-12
    dq, dk, dv, _ = mod.attention_backward(z, k, v, g, 0.6, True)
    for j in range(n):
        want = sum(g[i] / (i + 1) for i in range(j, n))
        assert np.max(np.abs(dv[j] - want)) < 1e-12
    # dK = scale * dS^T Q vanishes when Q = 0
    assert np.max(np.abs(dk)) < 1e-12


ALL_PINS = [
    pin_worked_example,
    pin_worked_example_exact,
    pin_brute_force,
    pin_brute_force_by_hand,
    pin_scipy,
    pin_probabilities,
    pin_blocked_equals_naive,
    pin_fp32_blocks,
    pin_closed_forms,
    pin_large_scores,
    pin_convex_hull,
    pin_shift_and_permutation,
    pin_rows_subset,
    pin_offsets_and_empty_rows,
    pin_decode_alignment,
    pin_split_kv,
    pin_backward_finite_differences,
    pin_backward_torch,
    pin_backward_invariants,
]
