"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded bf16 inputs.  Small cases compare every element; the five
measured workloads run at full size in the launch configuration bench.py
times and compare sampled (b, h) slices and rows."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_02_gb300.inputs import WORKLOADS, make_qkv, make_workload, sample_rows, sample_slices
from tests.parity import compare, log_stats, merge, within_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__ as entry
    entry.build()
    from exact_io_aware_02_gb300 import fa as mod
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    mod.fa_status(clear=True)
    return mod


def _np64(t):
    return t.to(torch.float64).numpy()


def run(fa, q, k, v, scale, causal):
    dev = torch.device("cuda")
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def check_slices(q, k, v, o, lse, scale, causal, slices, rows=None):
    stats = []
    for (b, h) in slices:
        ro, rl = oracle.naive_attention(_np64(q[b, h]), _np64(k[b, h]), _np64(v[b, h]), scale, causal, rows=rows)
        go = _np64(o[b, h]) if rows is None else _np64(o[b, h][rows])
        gl = _np64(lse[b, h]) if rows is None else _np64(lse[b, h][rows])
        stats.append(compare(go, gl, ro, rl))
    return merge(stats)


SMALL = [(B, H, N, d, causal)
         for (B, H, N) in ((1, 2, 128), (1, 1, 256), (2, 1, 384), (1, 2, 1000), (1, 1, 77), (1, 1, 1),
                           (1, 3, 640), (1, 1, 2049))
         for d in (64, 128) for causal in (False, True)]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL, ids=[f"B{a}H{b}N{c}d{e}{'c' if f else 'n'}" for a, b, c, e, f in SMALL])
def test_small_all_elements(fa, B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=1000 + N + d + int(causal))
    scale = 1.0 / math.sqrt(d)
    o, lse = run(fa, q, k, v, scale, causal)
    st = check_slices(q, k, v, o, lse, scale, causal, [(b, h) for b in range(B) for h in range(H)])
    assert within_tolerance(st), st


MHA_WORKLOADS = [n for n, w in WORKLOADS.items() if w.Hkv is None and w.Nk is None and w.direction == "fwd"]


@pytest.mark.parametrize("name", MHA_WORKLOADS)
def test_workload_full_size_sampled(fa, name):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o, lse = run(fa, q, k, v, w.scale, w.causal)
    n_slices = {"n128_d64": 1, "n2048_d64": 16, "causal_n8192_d128": 4,
                "wide_scores_n1024_d128": 32, "causal_n32768_d128": 4}[name]
    slices = sample_slices(w.B, w.H, n_slices, w.seed + 1)
    # every row of the sampled slices up to N = 8192; at N = 32768 the first two query
    # tiles (the rows that see the fewest keys) and 1792 sampled rows of each slice
    rows = None if w.N <= 8192 else sample_rows(w.N, 2048, w.seed + 2, leading=256)
    st = check_slices(q, k, v, o, lse, w.scale, w.causal, slices, rows)
    print(name, st)
    log_stats(name, st, slices, w.N if rows is None else len(rows))
    assert within_tolerance(st), st
    # properties over every output of the workload: finite, and O inside the V range per head
    og = o.to(torch.float32)
    assert torch.isfinite(og).all() and torch.isfinite(lse).all()
    vf = v.to(torch.float32)
    if not w.causal:
        lo = vf.amin(dim=2, keepdim=True)
        hi = vf.amax(dim=2, keepdim=True)
        slack = 1e-2 + 2.0 ** -8 * vf.abs().amax(dim=2, keepdim=True)
        assert bool(((og >= lo - slack) & (og <= hi + slack)).all())


def test_worked_example_replay(fa):
    """The hand-worked online-softmax example of the notes page (§8): scores
    (sqrt2, 1/sqrt2, 1/sqrt2) and v = (1, 0, 1), built from d = 64 vectors with
    scale 1/sqrt2; N = 3 exercises the ragged last tile."""
    q = torch.zeros(1, 1, 3, 64)
    k = torch.zeros(1, 1, 3, 64)
    v = torch.zeros(1, 1, 3, 64)
    q[0, 0, :, 0] = 1.0
    q[0, 0, :, 1] = 1.0
    k[0, 0, 0, :2] = 1.0
    k[0, 0, 1, 0] = 1.0
    k[0, 0, 2, 1] = 1.0
    v[0, 0, :, 0] = torch.tensor([1.0, 0.0, 1.0])
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / math.sqrt(2.0)
    o, lse = run(fa, q, k, v, scale, False)
    ro, rl = oracle.naive_attention(_np64(q[0, 0]), _np64(k[0, 0]), _np64(v[0, 0]), scale, False)
    st = compare(_np64(o[0, 0]), _np64(lse[0, 0]), ro, rl)
    assert within_tolerance(st), st
    # the page's printed result, 0.752, within its rounding plus the bf16 output's half ulp
    assert abs(float(o[0, 0, 0, 0]) - 0.752) <= 6e-4 + 2.0 ** -9


@pytest.mark.parametrize("c", [30.0, -30.0])
def test_large_constant_scores(fa, c):
    """Rows of +-30 scores: no overflow or NaN; O = mean of the V rows (causal:
    of the visible ones); LSE = score + ln(count)."""
    N, d = 384, 128
    scale = 1.0 / math.sqrt(d)
    a = float(torch.tensor(c / scale).to(torch.bfloat16))  # bf16 value with a*scale ~ c
    q = torch.zeros(1, 1, N, d)
    q[..., 0] = a
    k = torch.zeros(1, 1, N, d)
    k[..., 0] = 1.0
    _, _, v = make_qkv(1, 1, N, d, seed=42)
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run(fa, q, k, v, scale, causal)
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        ro, rl = oracle.naive_attention(_np64(q[0, 0]), _np64(k[0, 0]), _np64(v[0, 0]), scale, causal)
        st = compare(_np64(o[0, 0]), _np64(lse[0, 0]), ro, rl)
        assert within_tolerance(st), st
        s = a * scale
        cnt = np.arange(1, N + 1) if causal else np.full(N, N)
        assert np.max(np.abs(_np64(lse[0, 0]) - (s + np.log(cnt)))) <= 1e-3 * max(1.0, abs(s) + 6)


def test_near_uniform_attention(fa):
    """A scale near zero makes every visible key weigh the same: O is the mean of the visible
    V rows and LSE = ln(count) (plus a term of order scale * |q.k|)."""
    N, d = 700, 128
    q, k, v = make_qkv(1, 2, N, d, seed=91)
    scale = 1e-6
    for causal in (False, True):
        o, lse = run(fa, q, k, v, scale, causal)
        for h in range(2):
            ro, rl = oracle.naive_attention(_np64(q[0, h]), _np64(k[0, h]), _np64(v[0, h]), scale, causal)
            st = compare(_np64(o[0, h]), _np64(lse[0, h]), ro, rl)
            assert within_tolerance(st), st
            vv = _np64(v[0, h])
            mean = np.cumsum(vv, axis=0) / np.arange(1, N + 1)[:, None] if causal else np.broadcast_to(vv.mean(0), vv.shape)
            assert np.max(np.abs(_np64(o[0, h]) - mean)) <= 1e-2
            cnt = np.arange(1, N + 1) if causal else np.full(N, N)
            assert np.max(np.abs(_np64(lse[0, h]) - np.log(cnt))) <= 1e-3 * np.log(N) + 1e-3


def test_causal_row_zero_closed_form(fa):
    q, k, v = make_qkv(2, 2, 512, 128, seed=5)
    scale = 1.0 / math.sqrt(128)
    o, lse = run(fa, q, k, v, scale, True)
    for b in range(2):
        for h in range(2):
            assert torch.equal(o[b, h, 0], v[b, h, 0])   # one visible key: O = V[0] exactly
            want = scale * float((q[b, h, 0].double() * k[b, h, 0].double()).sum())
            assert abs(float(lse[b, h, 0]) - want) <= 1e-3 * max(1.0, abs(want))


def test_shift_invariance(fa):
    """Adding one vector to every K row leaves O unchanged (up to rounding) and
    shifts LSE_i by scale*q_i.u."""
    q, k, v = make_qkv(1, 2, 640, 64, seed=9)
    u = torch.zeros(64)
    u[3] = 2.0
    k2 = (k.float() + u).to(torch.bfloat16)
    scale = 0.125
    for causal in (False, True):
        o1, l1 = run(fa, q, k, v, scale, causal)
        o2, l2 = run(fa, q, k2, v, scale, causal)
        # k + u rounds to bf16, so the shifted scores differ slightly: check the shifted run
        # against the oracle on its own inputs, then the two outputs against each other
        ro, rl = oracle.naive_attention(_np64(q[0, 1]), _np64(k2[0, 1]), _np64(v[0, 1]), scale, causal)
        assert within_tolerance(compare(_np64(o2[0, 1]), _np64(l2[0, 1]), ro, rl))
        assert float((o1.float() - o2.float()).abs().max()) <= 2e-2


def test_argument_errors_on_device(fa):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 256, 128, seed=3))
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 256), 7.0, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    lib = fa.lib
    # host pointer for an input
    qh = q.cpu()
    assert lib.fa_fwd(qh.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      1, 1, 256, 128, 0.088, 0, s) == fa.FA_ERR_ARG
    # misaligned pointer, unsupported d, output aliasing an input
    assert lib.fa_fwd(q.data_ptr() + 2, k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      1, 1, 255, 128, 0.088, 0, s) == fa.FA_ERR_ARG
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      1, 1, 128, 256, 0.088, 0, s) == fa.FA_ERR_ARG
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), lse.data_ptr(),
                      1, 1, 256, 128, 0.088, 0, s) == fa.FA_ERR_ARG
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())   # nothing written


def test_stream_and_repeatability(fa):
    """Results are bitwise repeatable and independent of the stream used."""
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(2, 4, 1024, 128, seed=11))
    o1, l1 = fa.fa_fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = fa.fa_fwd(q, k, v, causal=True, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_status_word_clean(fa):
    assert fa.fa_status(clear=False) == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", ["all_large", "large_first_tile", "all_tiny", "tiny_later_tile"])
def test_v_outside_fp16_range(fa, case, d):
    """P V runs in fp16 with V held as fp16(v * 2^-K), K fixed per CTA by its first V tile:
    0 when that tile's largest |v| is in [2^-4, 65520), else chosen to bring it into
    [2^14, 2^15).  Uniformly large or tiny V, a large first tile before ordinary ones, and a
    tiny tile after ordinary ones are all exact.  Each case is checked against the oracle at
    V's own scale lam (power-of-two scalings of bf16 values are exact): |dO| / lam within the
    usual bounds, with the status word clean."""
    N = 640  # five K/V tiles
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(1, 2, N, d, seed=4100 + d + len(case))
    vf = v.float()
    lam = 1.0
    if case == "all_large":
        vf, lam = vf * 2.0 ** 20, 2.0 ** 20
    elif case == "large_first_tile":
        vf[..., :128, :] *= 2.0 ** 20
        lam = 2.0 ** 20
    elif case == "all_tiny":
        vf, lam = vf * 2.0 ** -30, 2.0 ** -30
    elif case == "tiny_later_tile":
        vf[..., 384:512, :] *= 2.0 ** -30
    v2 = vf.to(torch.bfloat16)
    assert torch.equal(v2.float(), vf)
    fa.fa_status(clear=True)
    for causal in (False, True):
        o, lse = run(fa, q, k, v2, scale, causal)
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        for h in range(2):
            ro, rl = oracle.naive_attention(_np64(q[0, h]), _np64(k[0, h]), _np64(v2[0, h]), scale, causal)
            st = compare(_np64(o[0, h]) / lam, _np64(lse[0, h]), ro / lam, rl)
            assert within_tolerance(st), (case, causal, h, st)
    assert fa.fa_status(clear=False) == 0


@pytest.mark.parametrize("case", ["large_later_tile", "tiny_first_tile"])
def test_v_tile_beyond_fp16_at_the_cta_scale_is_flagged(fa, case):
    """A V tile that fp16 cannot hold at the scale the CTA's first V tile fixed (a tile of
    values >= 65520 after ordinary ones; ordinary tiles after a tiny first tile) saturates,
    and the status word says so (FA_STATUS_V_RANGE); nothing faults, and the next call is
    clean."""
    N, d = 384, 128
    q, k, v = make_qkv(1, 1, N, d, seed=4202)
    vf = v.float()
    if case == "large_later_tile":
        vf[..., 256:384, :] *= 2.0 ** 20
    else:
        vf[..., :128, :] *= 2.0 ** -30
    fa.fa_status(clear=True)
    o, lse = run(fa, q, k, vf.to(torch.bfloat16), 1.0 / math.sqrt(d), False)
    assert torch.isfinite(lse).all()
    assert fa.fa_status(clear=True) & fa.FA_STATUS_V_RANGE
    q, k, v = make_qkv(1, 1, N, d, seed=4203)
    o, lse = run(fa, q, k, v, 1.0 / math.sqrt(d), False)
    assert fa.fa_status(clear=False) == 0
