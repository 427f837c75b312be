"""GPU parity of fa_fwd_fp8 (block-wise E4M3 attention with incoherent processing) against
the fp64 FP8 oracle (oracle/fp8.py), through the C ABI.

Two stages are checked.
* The quantisation, code by code: the workspace holds the E4M3 codes of Q', K' (rotated)
  and V (transposed) and their tile scales.  The kernel rotates in fp32 and the oracle in
  fp64, so a value that lies within fp32 rounding of an E4M3 tie may round the other way:
  every code must equal the oracle's or sit one E4M3 step from it, and nearly all must be
  equal.  Scales agree to fp32 rounding.
* The attention.  The oracle's reference is the exact attention of its dequantised Q', K'
  and V (fp8_attention); the kernel's one further rounding is P's, to E4M3 before the
  product with V.  The bounds come from the format alone: a term stored as an E4M3 value
  moves by at most half a step, 2^-4 of itself in the normal range and 2^-10 of the encoding
  scale below it, so the attention weight a_ij = p_ij / l_i moves by at most
  h_ij = max(2^-4 a_ij, 2^-10 / (sigma_j l_i)), sigma_j = 64 r_j the encoding scale of P's
  column j (the per-tile V scale over the largest one, reading R22).  Then, element by
  element, |dO| <= sum_j h_ij |v'_j| + half a bf16 ulp of O (the output's rounding); and,
  treating each rounding as uniform within its half step, the mean |dO| is held to 1.25 times
  the root-mean-square that model predicts.  LSE does not see P's rounding:
  |dLSE| <= 1e-3 max(1, |LSE|).  The oracle's own P-rounded variant (quantize_p=True, one
  plausible placement) is printed as a diagnostic only.
"""
import math

import numpy as np
import pytest
import torch

import oracle.attention as exact
import oracle.fp8 as f8
from exact_io_aware_02_gb300.inputs import (WORKLOADS, make_qkv, make_signs, make_workload, make_workload_signs,
                                            sample_rows, sample_slices)

from tests.parity import log_stats

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__ as entry
    entry.build()
    from exact_io_aware_02_gb300 import fa as mod
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    mod.fa_status(clear=True)
    return mod


def _np(t):
    return t.to(torch.float64).cpu().numpy()


def run(fa, q, k, v, signs, causal, scale=None):
    dev = torch.device("cuda")
    B, H, N, _ = q.shape
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, N, D), dtype=torch.uint8, device=dev)
    o, lse = fa.fa_fwd_fp8(q.to(dev), k.to(dev), v.to(dev), signs.to(dev), scale=scale, causal=causal,
                           workspace=ws)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu(), ws.cpu()


def decode_workspace(ws, B, H, N):
    """q8, k8 [BH, N_pad, 128], v8 [BH, N_pad, 128] (un-transposed) as floats; scales."""
    BH, n_pad = B * H, (N + 127) // 128 * 128
    T = n_pad // 128
    C = (BH * n_pad * D + 255) // 256 * 256
    SC = (BH * T * 4 + 255) // 256 * 256

    def codes(off, shape):
        return ws[off:off + BH * n_pad * D].view(torch.float8_e4m3fn).to(torch.float64).reshape(shape).numpy()
    q8 = codes(0, (BH, n_pad, D))
    k8 = codes(C, (BH, n_pad, D))
    v8 = codes(2 * C, (BH, D, n_pad)).transpose(0, 2, 1)

    def scales(off):
        return ws[off:off + BH * T * 4].view(torch.float32).to(torch.float64).reshape(BH, T).numpy()
    return q8, k8, v8, scales(3 * C), scales(3 * C + SC), scales(3 * C + 2 * SC)


def e4m3_step(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


def check_codes(got, want):
    equal = got == want
    near = np.abs(got - want) <= e4m3_step(np.maximum(np.abs(got), np.abs(want))) * (1 + 1e-9)
    return float(equal.mean()), bool(near.all())


CASES = [  # B, H, N, causal, qk_std
    (1, 2, 128, False, 1.0),
    (1, 2, 1000, True, 1.0),     # ragged last tile
    (2, 2, 2048, True, 1.0),
    (1, 2, 640, False, 3.0),     # sharp rows
    (1, 1, 1, True, 1.0),        # one row
    (1, 3, 129, False, 1.0),     # one row past a tile
]
IDS = ["b{}h{}n{}{}_std{}".format(b, h, n, "c" if c else "", int(s)) for b, h, n, c, s in CASES]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fp8_quantisation_matches_oracle(fa, case):
    B, H, N, causal, std = case
    q, k, v = make_qkv(B, H, N, D, seed=8100 + N, qk_std=std)
    signs = make_signs(D, 8200 + N)
    _, _, ws = run(fa, q, k, v, signs, causal)
    q8, k8, v8, sq, sk, sv = decode_workspace(ws, B, H, N)
    s = signs.numpy().astype(np.float64)
    n_pad = q8.shape[1]
    for bh in range(B * H):
        b, h = divmod(bh, H)
        for got, gs, src, rot in ((q8, sq, q, True), (k8, sk, k, True), (v8, sv, v, False)):
            x = _np(src[b, h])
            x = f8.rotate(x, s) if rot else x
            codes, scales = f8.quantize_blocks(x)
            assert np.allclose(gs[bh], scales, rtol=2e-6, atol=0)
            frac, near = check_codes(got[bh, :N], codes)
            assert near and frac > 0.995, (frac, near)
            assert not np.any(got[bh, N:n_pad])  # padding rows hold zero codes


def bf16_half_ulp(x):
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(ax, 2.0 ** -126))
    return np.ldexp(1.0, e - 9)


def p_rounding_bounds(qa, ka, va, s, scale, causal, rows=None):
    """The oracle's reference for one (b, h) slice and the format's bounds on P's rounding:
    (O_ref, LSE_ref, envelope, variance), envelope = H |V'|, variance = (H^2 / 3) V'^2."""
    qd, kd, vd = f8.fp8_inputs(qa, ka, va, s)
    ro, rl = exact.naive_attention(qd, kd, vd, scale, causal, rows=rows)
    nk = kd.shape[0]
    r = np.arange(qd.shape[0]) if rows is None else np.asarray(rows)
    sc = scale * (qd[r] @ kd.T)
    if causal:
        sc = np.where(np.arange(nk)[None, :] > r[:, None], -np.inf, sc)
    p = np.exp(sc - sc.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    _, sv = f8.quantize_blocks(np.asarray(va, dtype=np.float64))
    sigma = 64.0 * np.repeat(sv / sv.max(), f8.BLOCK_ROWS)[:nk]
    h = np.where(p > 0.0, np.maximum(2.0 ** -4 * p / l, 2.0 ** -10 / (sigma[None, :] * l)), 0.0)
    return ro, rl, h @ np.abs(vd), (h * h / 3.0) @ (vd * vd)


def fp8_stats(o, lse, q, k, v, signs, causal, scale, heads, rows=None):
    s = signs.numpy().astype(np.float64)
    over, d_sum, d_max, n, var_sum, lse_err, m_max = -np.inf, 0.0, 0.0, 0, 0.0, 0.0, 0.0
    for b, h in heads:
        qa, ka, va = _np(q[b, h]), _np(k[b, h]), _np(v[b, h])
        ro, rl, env, var = p_rounding_bounds(qa, ka, va, s, scale, causal, rows)
        go = _np(o[b, h]) if rows is None else _np(o[b, h])[rows]
        gl = _np(lse[b, h]) if rows is None else _np(lse[b, h])[rows]
        assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
        d = np.abs(go - ro)
        half = bf16_half_ulp(ro)
        over = max(over, float(np.max(d - (env + half + 1e-4))))
        d_sum += float(d.sum())
        d_max = max(d_max, float(d.max()))
        n += d.size
        var_sum += float((var + half * half / 3.0).sum())
        lse_err = max(lse_err, float(np.max(np.abs(gl - rl) / np.maximum(1.0, np.abs(rl)))))
        mo, _ = f8.fp8_attention(qa, ka, va, scale, causal, s, rows=rows, quantize_p=True)
        m_max = max(m_max, float(np.abs(mo - ro).max()))
    return {"over_envelope": over, "d_mean": d_sum / n, "d_max": d_max, "rms_model": float(np.sqrt(var_sum / n)),
            "lse": lse_err, "replay_max_diagnostic": m_max}


def within(st):
    return st["over_envelope"] <= 0.0 and st["d_mean"] <= 1.25 * st["rms_model"] and st["lse"] <= 1e-3


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fp8_attention_parity(fa, case):
    B, H, N, causal, std = case
    q, k, v = make_qkv(B, H, N, D, seed=8100 + N, qk_std=std)
    signs = make_signs(D, 8200 + N)
    scale = 1.0 / math.sqrt(D)
    o, lse, _ = run(fa, q, k, v, signs, causal)
    st = fp8_stats(o, lse, q, k, v, signs, causal, scale, [(b, h) for b in range(B) for h in range(H)])
    print(case, st)
    log_stats("fp8_" + "_".join(str(x) for x in case), st, [(b, h) for b in range(B) for h in range(H)], N)
    assert within(st), st


def test_fp8_close_to_exact_attention(fa):
    """Against exact (bf16-input) attention: the kernel's RMSE is at most the FP8 reference's own
    (the error of quantising Q', K' and V, which the oracle measures directly) plus the
    root-mean-square the format predicts for P's rounding and the bf16 output (the triangle
    inequality).  The oracle's P-rounded variant is printed for comparison only."""
    B, H, N = 1, 2, 1024
    q, k, v = make_qkv(B, H, N, D, seed=8301)
    signs = make_signs(D, 8302)
    o, _, _ = run(fa, q, k, v, signs, True)
    s = signs.numpy().astype(np.float64)
    for h in range(H):
        qa, ka, va = _np(q[0, h]), _np(k[0, h]), _np(v[0, h])
        oe, _ = exact.naive_attention(qa, ka, va, 1 / math.sqrt(D), True)
        ro, _, _, var = p_rounding_bounds(qa, ka, va, s, 1 / math.sqrt(D), True)
        om, _ = f8.fp8_attention(qa, ka, va, 1 / math.sqrt(D), True, s, quantize_p=True)
        rmse_k = float(np.sqrt(np.mean((_np(o[0, h]) - oe) ** 2)))
        rmse_ref = float(np.sqrt(np.mean((ro - oe) ** 2)))
        half = bf16_half_ulp(ro)
        rms_p = float(np.sqrt(np.mean(var + half * half / 3.0)))
        print("rmse kernel", rmse_k, "reference", rmse_ref, "P model", rms_p,
              "replay (diagnostic)", float(np.sqrt(np.mean((om - oe) ** 2))))
        assert rmse_k <= rmse_ref + 1.25 * rms_p


FP8_WORKLOADS = [n for n, w in WORKLOADS.items() if w.direction == "fp8"]


@pytest.mark.parametrize("name", FP8_WORKLOADS)
def test_fp8_workload_full_size_sampled(fa, name):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    signs = make_workload_signs(w)
    o, lse, _ = run(fa, q, k, v, signs, w.causal)
    heads = sample_slices(w.B, w.H, 2, w.seed + 1)
    rows = sample_rows(w.N, 256, w.seed + 2)
    st = fp8_stats(o, lse, q, k, v, signs, w.causal, w.scale, heads, rows)
    print(name, st)
    log_stats(name, st, heads, len(rows))
    assert within(st), st
    assert torch.isfinite(o.to(torch.float32)).all() and torch.isfinite(lse).all()
    assert fa.fa_status(clear=False) == 0


def test_fp8_repeatable_and_status_clean(fa):
    q, k, v = make_qkv(1, 2, 700, D, seed=8401)
    signs = make_signs(D, 8402)
    a = run(fa, q, k, v, signs, True)
    b = run(fa, q, k, v, signs, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert fa.fa_status(clear=False) == 0


def test_fp8_argument_errors(fa):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 256, D, seed=8501))
    signs = make_signs(D, 8502).to(dev)
    o = torch.full_like(q, 5.0)
    lse = torch.full((1, 1, 256), 5.0, device=dev)
    need = fa.fa_fwd_fp8_workspace_bytes(1, 1, 256, D)
    assert fa.fa_fwd_fp8_workspace_bytes(1, 1, 256, 64) == 0
    ws = torch.empty(need + 512, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError):  # workspace too small
        fa.fa_fwd_fp8(q, k, v, signs, o, lse, workspace=ws[: need - 256])
    with pytest.raises(fa.FAError):  # workspace not 256-byte aligned
        fa.fa_fwd_fp8(q, k, v, signs, o, lse, workspace=ws[16: need + 16])
    with pytest.raises(fa.FAError):  # d = 64 is not supported
        q64 = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device=dev)
        fa.fa_fwd_fp8(q64, q64.clone(), q64.clone(), signs, workspace=ws)
    with pytest.raises(fa.FAError):  # output overlaps the workspace
        fa.fa_fwd_fp8(q, k, v, signs, ws[:256 * D * 2].view(torch.bfloat16).view(1, 1, 256, D), lse,
                      workspace=ws)
    torch.cuda.synchronize()
    assert bool((o == 5.0).all()) and bool((lse == 5.0).all())


@pytest.mark.parametrize("groups_per_chunk", [0, 1, 3])
def test_fp8_host_equals_device_call(fa, groups_per_chunk):
    """fa_fwd_fp8_host runs fa_fwd_fp8's kernels per chunk of heads: bitwise the same O, LSE."""
    dev = torch.device("cuda")
    B, H, N = 2, 3, 700
    q, k, v = make_qkv(B, H, N, D, seed=8601)
    signs = make_signs(D, 8602).to(dev)
    need = fa.fa_fwd_fp8_workspace_bytes(B, H, N, D)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    o_ref, l_ref = fa.fa_fwd_fp8(q.to(dev), k.to(dev), v.to(dev), signs, causal=True, workspace=ws)
    torch.cuda.synchronize()
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.full(q.shape, 7.0, dtype=torch.bfloat16).pin_memory()
    lh = torch.full((B, H, N), 7.0, dtype=torch.float32).pin_memory()
    qd, kd, vd = (torch.zeros(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v))
    od = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ld = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws2 = torch.empty(need, dtype=torch.uint8, device=dev)
    fa.fa_fwd_fp8_host(qh, kh, vh, oh, lh, qd, kd, vd, signs, od, ld, ws2, causal=True,
                       groups_per_chunk=groups_per_chunk)
    torch.cuda.synchronize()
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())
    assert fa.fa_status(clear=False) == 0


def test_fp8_host_one_stream_when_workspace_is_tight(fa):
    """A workspace that holds one chunk's layout but not two runs the chunks on one stream."""
    dev = torch.device("cuda")
    B, H, N = 1, 2, 256
    q, k, v = make_qkv(B, H, N, D, seed=8701)
    signs = make_signs(D, 8702).to(dev)
    need = fa.fa_fwd_fp8_workspace_bytes(B, H, N, D)
    o_ref, l_ref = fa.fa_fwd_fp8(q.to(dev), k.to(dev), v.to(dev), signs, causal=False)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    qd, kd, vd = (torch.zeros(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v))
    od = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ld = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)  # holds two 1-head parts at most
    fa.fa_fwd_fp8_host(qh, kh, vh, oh, lh, qd, kd, vd, signs, od, ld, ws, causal=False, groups_per_chunk=2)
    torch.cuda.synchronize()
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())
