"""Pins of the FP8 oracle (oracle/fp8.py) to facts outside it: the E4M3 bit layout,
torch's own float8_e4m3fn conversion, the algebra of the Hadamard rotation, a small
case worked by hand, bounds that follow from the format, and the pages' claim that
incoherent processing lowers the FP8 attention error ([P2] §10 ③, §12.2).

Each pin takes the module under test, so that tests/test_oracle_mutants.py can run
the same pins against planted mistakes."""
from __future__ import annotations

import math

import numpy as np

import oracle.attention as exact


def _rng(seed):
    return np.random.default_rng(1000 + seed)


def pin_e4m3_table(mod):
    """127 finite non-negative values: 0, seven subnormals k/8 * 2^-6, then 15 binades of
    eight values each, except that the top binade has no 1.875 * 2^8 (that code is NaN).
    Largest 448, smallest normal 2^-6, smallest subnormal 2^-9."""
    t = mod.e4m3_values()
    assert t.shape == (127,)
    assert np.all(np.diff(t) > 0)
    assert t[0] == 0.0 and t[1] == 2.0 ** -9 and t[7] == 7 * 2.0 ** -9 and t[8] == 2.0 ** -6
    assert t[-1] == 448.0 and t[-2] == 416.0
    assert t[8 + 8 * 7] == 2.0 ** 1  # 2.0 is code 0x48


def pin_e4m3_matches_torch(mod):
    """Round to nearest even, as torch.float8_e4m3fn does, over the finite range, for
    float32 inputs (the kernel converts from fp32; torch converts fp64 through fp32, so it
    is compared on fp32 values): random values, every representable value, every midpoint
    and the float32 values just beside them."""
    import torch
    t = mod.e4m3_values().astype(np.float32)
    mids = ((t[1:].astype(np.float64) + t[:-1]) / 2).astype(np.float32)  # exact in fp32
    rng = _rng(1)
    xs = np.concatenate([
        t, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
        rng.uniform(0, 448, 4000).astype(np.float32),
        np.exp(rng.uniform(np.log(1e-4), np.log(448), 4000)).astype(np.float32),
    ]).astype(np.float32)
    xs = xs[xs <= 448.0]
    xs = np.concatenate([xs, -xs])
    want = torch.tensor(xs, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mod.e4m3_round(xs.astype(np.float64))
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]


def pin_e4m3_saturation(mod):
    """Finite values beyond 448 saturate (the kernel's cvt ... satfinite), sign kept."""
    xs = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 1e6, 1e300])
    assert np.all(mod.e4m3_round(xs) == 448.0)
    assert np.all(mod.e4m3_round(-xs) == -448.0)
    assert mod.e4m3_round(np.array([0.0]))[0] == 0.0


def pin_rotation_by_hand(mod):
    """d = 2, x = (1, 2), signs (+1, -1): x*s = (1, -2); H2 = [[1, 1], [1, -1]] gives
    (1 - 2, 1 + 2) = (-1, 3); over sqrt(2): (-0.7071..., 2.1213...).  d = 4, x = e_0 * 8:
    every coordinate becomes +-8/2 = +-4 with signs s_0 * (row 0 of H4) = s_0 * (1, 1, 1, 1)."""
    got = mod.rotate(np.array([[1.0, 2.0]]), np.array([1.0, -1.0]))
    assert np.allclose(got, [[-1 / np.sqrt(2), 3 / np.sqrt(2)]], rtol=0, atol=1e-15)
    got = mod.rotate(np.array([[8.0, 0.0, 0.0, 0.0]]), np.array([-1.0, 1.0, 1.0, -1.0]))
    assert np.allclose(got, [[-4.0, -4.0, -4.0, -4.0]], rtol=0, atol=1e-15)
    h4 = mod.hadamard(4)
    assert np.array_equal(h4, [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]])


def pin_rotation_preserves_scores(mod):
    """H H^T = d I, so the rotation keeps every dot product and norm; a single large
    coordinate is spread evenly over all d coordinates (incoherence)."""
    rng = _rng(2)
    for d in (1, 2, 8, 64, 128):
        h = mod.hadamard(d)
        assert np.array_equal(h @ h.T, d * np.eye(d))
        q, k = rng.standard_normal((5, d)), rng.standard_normal((7, d))
        s = rng.choice([-1.0, 1.0], d)
        qr, kr = mod.rotate(q, s), mod.rotate(k, s)
        assert np.max(np.abs(qr @ kr.T - q @ k.T)) < 1e-12
        assert np.max(np.abs(np.linalg.norm(qr, axis=1) - np.linalg.norm(q, axis=1))) < 1e-12
        spike = np.zeros((1, d))
        spike[0, d // 2] = 50.0
        assert np.allclose(np.abs(mod.rotate(spike, s)), 50.0 / np.sqrt(d), rtol=0, atol=1e-12)


def pin_quantize_bounds(mod):
    """Per tile: the largest magnitude maps to +-448 exactly; every element is within half
    an E4M3 step of x / s (relative 2^-4 for normals, 2^-10 absolute for subnormals);
    an all-zero tile has scale 1; a ragged last tile has its own scale."""
    rng = _rng(3)
    x = rng.standard_normal((300, 16)) * np.repeat(rng.uniform(0.01, 50, 3), 100)[:, None]
    codes, scales = mod.quantize_blocks(x, 128)
    assert scales.shape == (3,)
    for t in range(3):
        blk = x[t * 128:(t + 1) * 128]
        assert abs(scales[t] - np.abs(blk).max() / 448.0) <= 1e-15 * scales[t]
        c = codes[t * 128:(t + 1) * 128]
        assert np.max(np.abs(c)) == 448.0
        y = blk / scales[t]
        bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10)
        assert np.all(np.abs(c - y) <= bound + 1e-12)
    z_codes, z_scales = mod.quantize_blocks(np.zeros((10, 4)), 128)
    assert z_scales[0] == 1.0 and not np.any(z_codes)
    deq = mod.dequantize_blocks(codes, scales, 128)
    assert deq.shape == x.shape and np.max(np.abs(deq - x) / np.abs(x).max()) < 2 ** -4


def pin_fp8_exact_when_representable(mod):
    """Without rotation, inputs already of the form (tile scale) x (E4M3 values, tile max
    448) quantise exactly, so FP8 attention equals exact attention."""
    rng = _rng(4)
    t = mod.e4m3_values()
    n, d = 200, 8

    def representable():
        x = rng.choice(np.concatenate([t, -t]), size=(n, d))
        x[0, 0] = 448.0
        x[128, 0] = 448.0
        return x * 0.01
    q, k, v = representable(), representable(), representable()
    for causal in (False, True):
        o8, l8 = mod.fp8_attention(q, k, v, 0.05, causal, np.ones(d), rotate_qk=False)
        o, l = exact.naive_attention(q, k, v, 0.05, causal)
        assert np.max(np.abs(o8 - o)) < 1e-12 and np.max(np.abs(l8 - l)) < 1e-12


def pin_incoherent_processing_helps(mod):
    """[P2] §12.2: with outlier channels in Q and K (a few coordinates 20x larger, as in
    trained models), rotating before quantisation lowers the FP8 attention error against
    exact attention, here by more than 1.5x; on plain normal inputs it does not hurt."""
    rng = _rng(5)
    n, d = 512, 128
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    out = rng.choice(d, 4, replace=False)
    q[:, out] *= 20.0
    k[:, out] *= 20.0
    scale = 1.0 / np.sqrt(d) / 8.0
    o, _ = exact.naive_attention(q, k, v, scale, True)
    s = rng.choice([-1.0, 1.0], d)

    def rmse(rot):
        o8, _ = mod.fp8_attention(q, k, v, scale, True, s, rotate_qk=rot)
        return np.sqrt(np.mean((o8 - o) ** 2))
    plain, rotated = rmse(False), rmse(True)
    assert rotated * 1.5 < plain, (plain, rotated)
    q2, k2, v2 = (rng.standard_normal((n, d)) for _ in range(3))
    o2, _ = exact.naive_attention(q2, k2, v2, 1 / np.sqrt(d), False)
    e_plain = np.sqrt(np.mean((mod.fp8_attention(q2, k2, v2, 1 / np.sqrt(d), False, s, rotate_qk=False)[0] - o2) ** 2))
    e_rot = np.sqrt(np.mean((mod.fp8_attention(q2, k2, v2, 1 / np.sqrt(d), False, s, rotate_qk=True)[0] - o2) ** 2))
    assert e_rot < 1.3 * e_plain


def pin_quantized_p_is_close(mod):
    """Rounding P to E4M3 (before the product with V) moves O by a few percent of |V| at
    most and leaves LSE untouched; with P exact the two agree to rounding."""
    rng = _rng(6)
    n, d = 300, 64
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    s = rng.choice([-1.0, 1.0], d)
    o, l = mod.fp8_attention(q, k, v, 1 / 8.0, True, s)
    oq, lq = mod.fp8_attention(q, k, v, 1 / 8.0, True, s, quantize_p=True)
    assert np.max(np.abs(lq - l)) < 1e-12
    assert np.max(np.abs(oq - o)) < 0.1 * np.abs(v).max()
    assert np.mean(np.abs(oq - o)) < 0.01 * np.abs(v).max()


def pin_quantized_p_worked_by_hand(mod):
    """P rounded to E4M3 on a case worked by hand (the reading: each term p_j, taken against
    the row max, is stored as e4m3(p_j * 64 * r_j), r_j = key j's V-tile scale over the
    largest V-tile scale, and used as that value / (64 r_j); l and LSE use the unrounded p).

    One query q = (1, 1), scale 1, no rotation, 2-row tiles.  Keys (1,1), (1,0), (0,1),
    (-3.5,-3.5) give scores 2, 1, 1, -7, so p = (1, e^-1, e^-1, e^-9).  Every Q, K and V value
    is exact after its tile's quantisation (codes 448, 224, 128, 0), so only P is rounded.
    V rows (3,0), (1.5,3) | (1,0.5), (0,1): V-tile maxima 3 and 1, so r = (1, 1, 1/3, 1/3).
      x_0 = 64                      -> 64                      p~_0 = 1
      x_1 = 64/e     = 23.544 (step 2 in [16,32))   -> 24      p~_1 = 24/64 = 0.375
      x_2 = 64/(3e)  = 7.8481 (step 0.5 in [4,8))   -> 8       p~_2 = 8*3/64 = 0.375
      x_3 = 64e^-9/3 = 0.0026327 (subnormal, step 2^-9 = 0.0019531: 1.348 steps) -> 2^-9
                                                               p~_3 = 3 * 2^-15
    l = 1 + 2/e + e^-9 = 1.7358823; O = (3 + 0.5625 + 0.375, 1.125 + 0.1875 + 3*2^-15) / l
      = (2.2682990, 0.7561524); LSE = 2 + ln l.
    A power-of-two change of the gain moves no normal-range rounding (E4M3 is scale-free there)
    but does move the subnormal x_3, and a ratio that is not sv_j / max sv changes x_3 too."""
    q = np.array([[1.0, 1.0]])
    k = np.array([[1.0, 1.0], [1.0, 0.0], [0.0, 1.0], [-3.5, -3.5]])
    v = np.array([[3.0, 0.0], [1.5, 3.0], [1.0, 0.5], [0.0, 1.0]])
    o, lse = mod.fp8_attention(q, k, v, 1.0, False, np.ones(2), rotate_qk=False, quantize_p=True,
                               block_rows=2)
    l = 1.0 + 2.0 * math.exp(-1.0) + math.exp(-9.0)
    want = np.array([3.0 + 0.5625 + 0.375, 1.125 + 0.1875 + 3.0 * 2.0 ** -15]) / l
    assert abs(l - 1.7358823) < 1e-7
    assert np.max(np.abs(o[0] - want)) < 1e-12, (o, want)
    assert np.max(np.abs(o[0] - np.array([2.2682990, 0.7561524]))) < 1e-7
    assert abs(lse[0] - (2.0 + math.log(l))) < 1e-12
    # with P exact the same inputs give the plain softmax average
    o_exact, _ = mod.fp8_attention(q, k, v, 1.0, False, np.ones(2), rotate_qk=False, block_rows=2)
    pe = np.exp(np.array([0.0, -1.0, -1.0, -9.0]))
    assert np.max(np.abs(o_exact[0] - pe @ v / l)) < 1e-12


def pin_p_rounding_within_format_bound(mod):
    """Each rounded term of the quantize_p branch differs from p by at most half an E4M3 step:
    2^-4 p where p * 64 * r is a normal E4M3 value, 2^-10 / (64 r) below (subnormal step
    2^-9).  Checked term by term through one-key rows (O = v~ p~ / l with v = 1)."""
    rng = _rng(7)
    for t in range(200):
        s = -rng.uniform(0.0, 14.0)           # second key's score below the first (0)
        ratio_tile = rng.uniform(1.0, 6.0)     # first V tile's scale over the second's
        q = np.array([[1.0, 0.0]])
        k = np.array([[0.0, 0.0], [s, 0.0]])
        v = np.array([[ratio_tile, 0.0], [0.0, 1.0]])   # key 1's column-1 value 1, r_1 = 1/ratio_tile
        o, _ = mod.fp8_attention(q, k, v, 1.0, False, np.ones(2), rotate_qk=False, quantize_p=True,
                                 block_rows=1)
        vd = mod.fp8_inputs(q, k, v, np.ones(2), rotate_qk=False, block_rows=1)[2]
        p1 = math.exp(float(mod.fp8_inputs(q, k, v, np.ones(2), rotate_qk=False, block_rows=1)[1][1, 0]))
        l = 1.0 + p1
        p1_rounded = o[0, 1] * l / vd[1, 1]
        r1 = 1.0 / ratio_tile
        bound = max(2.0 ** -4 * p1, 2.0 ** -10 / (64.0 * r1))
        assert abs(p1_rounded - p1) <= bound * (1 + 1e-9), (s, ratio_tile, p1, p1_rounded, bound)


FP8_PINS = [
    pin_e4m3_table,
    pin_e4m3_matches_torch,
    pin_e4m3_saturation,
    pin_rotation_by_hand,
    pin_rotation_preserves_scores,
    pin_quantize_bounds,
    pin_fp8_exact_when_representable,
    pin_incoherent_processing_helps,
    pin_quantized_p_is_close,
    pin_quantized_p_worked_by_hand,
    pin_p_rounding_within_format_bound,
]
