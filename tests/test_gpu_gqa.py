"""GPU parity of fa_fwd_gqa (grouped K/V heads, different query/key lengths with the
bottom-right causal mask, split-K/V) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_02_gb300.inputs import WORKLOADS, make_qkv_gqa, make_workload, sample_slices
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


def run(fa, q, k, v, scale, causal, n_splits):
    dev = torch.device("cuda")
    o, lse = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal, n_splits=n_splits)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def check(q, k, v, o, lse, scale, causal, heads=None, rows=None):
    B, Hq, Nq, _ = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    heads = heads or [(b, h) for b in range(B) for h in range(Hq)]
    stats = []
    for b, h in heads:
        ro, rl = oracle.naive_attention(_np64(q[b, h]), _np64(k[b, h // G]), _np64(v[b, h // G]),
                                        scale, causal, rows=rows, q_offset=Nk - Nq)
        go = _np64(o[b, h]) if rows is None else _np64(o[b, h][rows])
        gl = _np64(lse[b, h]) if rows is None else _np64(lse[b, h][rows])
        stats.append(compare(go, gl, ro, rl))
    return merge(stats)


CASES = [  # B, Hq, Hkv, Nq, Nk, d, causal, n_splits
    (1, 4, 2, 200, 200, 128, True, 1),     # GQA prefill, square causal
    (1, 8, 1, 64, 64, 64, False, 1),       # MQA
    (2, 8, 2, 1, 1000, 128, False, 4),     # decoding, split keys
    (2, 8, 2, 1, 1000, 128, True, 4),      # one query at the end: causal = all keys
    (1, 4, 4, 3, 777, 64, True, 3),        # a few new queries, bottom-right mask, ragged
    (1, 2, 2, 100, 300, 128, True, 1),     # fewer queries than keys
    (1, 2, 1, 300, 100, 64, True, 2),      # more queries than keys: early rows see nothing
    (1, 2, 2, 2, 200, 128, False, 8),      # more splits than key tiles: empty splits
    (1, 6, 3, 130, 513, 128, False, 5),    # query tiles straddling heads
    (1, 32, 8, 1, 4096, 128, False, 16),   # long decode
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,n_splits", CASES,
                         ids=[f"B{a}Hq{b}Hkv{c}Nq{e}Nk{f}d{g}{'c' if h else 'n'}s{i}" for a, b, c, e, f, g, h, i in CASES])
def test_gqa_all_elements(fa, B, Hq, Hkv, Nq, Nk, d, causal, n_splits):
    q, k, v = make_qkv_gqa(B, Hq, Hkv, Nq, Nk, d, seed=3000 + Nq + Nk + d + n_splits)
    scale = 1.0 / math.sqrt(d)
    o, lse = run(fa, q, k, v, scale, causal, n_splits)
    st = check(q, k, v, o, lse, scale, causal)
    assert within_tolerance(st), st


def test_mha_special_case_matches_fa_fwd(fa):
    """fa_fwd_gqa with Hq = Hkv, Nq = Nk, one split is fa_fwd, bit for bit."""
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv_gqa(2, 4, 4, 640, 640, 128, seed=77))
    for causal in (False, True):
        o1, l1 = fa.fa_fwd(q, k, v, causal=causal)
        o2, l2 = fa.fa_fwd_gqa(q, k, v, causal=causal, n_splits=1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_count_changes_only_rounding(fa):
    q, k, v = make_qkv_gqa(1, 8, 2, 1, 3000, 128, seed=78)
    scale = 1.0 / math.sqrt(128)
    base = None
    for n_splits in (1, 2, 7, 24):
        o, lse = run(fa, q, k, v, scale, False, n_splits)
        st = check(q, k, v, o, lse, scale, False)
        assert within_tolerance(st), (n_splits, st)
        if base is None:
            base = (o.float(), lse)
        else:
            assert float((o.float() - base[0]).abs().max()) <= 2e-2
            assert float((lse - base[1]).abs().max()) <= 1e-3


def test_workspace_errors(fa):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv_gqa(1, 4, 2, 1, 512, 128, seed=79))
    o = torch.empty_like(q)
    lse = torch.empty((1, 4, 1), device=dev)
    need = fa.fa_fwd_gqa_workspace_bytes(1, 4, 1, 128, 4)
    assert need > 0 and fa.fa_fwd_gqa_workspace_bytes(1, 4, 1, 128, 1) == 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    lib = fa.lib
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 4, 2, 1, 512, 128,
            0.088, 0)
    assert lib.fa_fwd_gqa(*args, 4, small.data_ptr(), small.numel(), s) == fa.FA_ERR_ARG
    assert lib.fa_fwd_gqa(*args, 4, None, 0, s) == fa.FA_ERR_ARG
    assert lib.fa_fwd_gqa(*args, 0, None, 0, s) == fa.FA_ERR_ARG
    bad_heads = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 4, 3, 1, 512, 128,
                 0.088, 0, 1, None, 0, s)
    assert lib.fa_fwd_gqa(*bad_heads) == fa.FA_ERR_ARG


@pytest.mark.parametrize("name", ["gqa_causal_n8192_d128", "gqa_decode_nk32768_d128"])
def test_gqa_workload_full_size_sampled(fa, name):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o, lse = run(fa, q, k, v, w.scale, w.causal, w.n_splits)
    heads = sample_slices(w.B, w.H, 8, w.seed + 1)
    st = check(q, k, v, o, lse, w.scale, w.causal, heads=heads)   # every row of 8 query heads
    print(name, st)
    log_stats(name, st, heads, w.N)
    assert within_tolerance(st), st
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_status_word_clean_after_gqa(fa):
    assert fa.fa_status(clear=False) == 0


def test_split_kv_v_beyond_fp16_is_flagged(fa):
    """Split-K/V with several query tiles runs the fp16 P V instance and writes fp32 partials:
    a V tile fp16 cannot hold at the CTA's scale is flagged there too (FA_STATUS_V_RANGE), and
    ordinary V on the same shape is exact and clean."""
    q, k, v = make_qkv_gqa(1, 4, 2, 300, 1024, 128, seed=3301)
    scale = 1.0 / math.sqrt(128)
    fa.fa_status(clear=True)
    o, lse = run(fa, q, k, v, scale, False, 3)
    assert within_tolerance(check(q, k, v, o, lse, scale, False))
    assert fa.fa_status(clear=True) == 0
    vf = v.float()
    vf[:, :, 640:768, :] *= 2.0 ** 20          # a K/V tile of the second split
    o, lse = run(fa, q, k, vf.to(torch.bfloat16), scale, False, 3)
    assert torch.isfinite(lse).all()
    assert fa.fa_status(clear=True) & fa.FA_STATUS_V_RANGE
