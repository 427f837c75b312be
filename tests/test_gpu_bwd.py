"""GPU parity of fa_bwd (dQ, dK, dV with S and P recomputed from the forward's LSE)
against the fp64 oracle, through the C ABI.

The backward consumes the forward's own O and LSE (that is how it is used), so each
case runs fa_fwd_gqa first.  The oracle recomputes everything in fp64 from the bf16
inputs; for grouped K/V heads the gradient of a shared K/V head is the sum of the
oracle's per-query-head gradients.  Tolerances: tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_02_gb300.inputs import WORKLOADS, make_dout, make_qkv_gqa, make_workload, make_workload_dout
from tests.parity import grad_compare, grad_within_tolerance

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
    return t.to(torch.float64).cpu().numpy()


def run(fa, q, k, v, do, causal, scale=None):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_gqa(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv, delta = fa.fa_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal)
    torch.cuda.synchronize()
    return dq.cpu(), dk.cpu(), dv.cpu(), delta.cpu()


def oracle_grads(q, k, v, do, scale, causal, kv_heads):
    """Oracle gradients for the K/V heads ``kv_heads`` [(b, g)]: dQ and D of every
    query head of the group, dK and dV summed over the group."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    out = {}
    for b, g in kv_heads:
        dk_sum = dv_sum = 0.0
        dqs, ds = [], []
        for h in range(g * G, (g + 1) * G):
            dq, dk, dv, d_row = oracle.attention_backward(_np64(q[b, h]), _np64(k[b, g]), _np64(v[b, g]),
                                                          _np64(do[b, h]), scale, causal)
            dk_sum = dk_sum + dk
            dv_sum = dv_sum + dv
            dqs.append(dq)
            ds.append(d_row)
        out[(b, g)] = (np.stack(dqs), dk_sum, dv_sum, np.stack(ds))
    return out


def check(q, k, v, do, res, scale, causal, kv_heads=None):
    dq, dk, dv, delta = res
    B, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    G = Hq // Hkv
    kv_heads = kv_heads or [(b, g) for b in range(B) for g in range(Hkv)]
    ref = oracle_grads(q, k, v, do, scale, causal, kv_heads)
    got = {n: [] for n in ("dq", "dk", "dv", "delta")}
    want = {n: [] for n in ("dq", "dk", "dv", "delta")}
    for (b, g), (rdq, rdk, rdv, rd) in ref.items():
        got["dq"].append(_np64(dq[b, g * G:(g + 1) * G]))
        want["dq"].append(rdq)
        got["dk"].append(_np64(dk[b, g]))
        want["dk"].append(rdk)
        got["dv"].append(_np64(dv[b, g]))
        want["dv"].append(rdv)
        got["delta"].append(_np64(delta[b, g * G:(g + 1) * G]))
        want["delta"].append(rd)
    return {n: grad_compare(np.concatenate([x.ravel() for x in got[n]]),
                            np.concatenate([x.ravel() for x in want[n]])) for n in got}


def case_stats_line(stats):
    return " ".join("{}:{:.2e}/{:.2e}".format(n, st["max_rel"], st["mean_rel"]) for n, st in stats.items())


CASES = [  # B, Hq, Hkv, N, d, causal
    (1, 2, 2, 128, 128, False),    # one tile
    (1, 2, 2, 256, 64, True),      # two tiles, causal diagonal
    (1, 2, 2, 1000, 128, True),    # ragged last tile
    (1, 2, 2, 640, 128, False),    # five tiles
    (1, 4, 2, 77, 64, False),      # grouped heads, query tiles straddle heads
    (2, 4, 1, 300, 128, True),     # one K/V head for four query heads, ragged
    (1, 1, 1, 1, 64, True),        # a single row
    (1, 3, 3, 129, 64, True),      # one row past a tile
    (1, 8, 2, 384, 128, True),     # four query heads per K/V head, causal
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}_hq{}_hkv{}_n{}_d{}_{}".format(
    *c[:5], "causal" if c[5] else "full"))
def test_bwd_parity(fa, case):
    B, Hq, Hkv, N, d, causal = case
    q, k, v = make_qkv_gqa(B, Hq, Hkv, N, N, d, seed=4100 + N + d)
    do = make_dout(q.shape, seed=4200 + N + d)
    scale = 1.0 / d ** 0.5
    stats = check(q, k, v, do, run(fa, q, k, v, do, causal), scale, causal)
    print(case_stats_line(stats))
    for name, st in stats.items():
        assert grad_within_tolerance(st), (name, st)


def test_bwd_wide_scores(fa):
    """Score std 3 (sharp rows): the case with the largest rounding error."""
    q, k, v = make_qkv_gqa(1, 2, 2, 512, 512, 128, seed=4301, qk_std=3.0)
    do = make_dout(q.shape, seed=4302)
    stats = check(q, k, v, do, run(fa, q, k, v, do, False), 1 / 128 ** 0.5, False)
    print(case_stats_line(stats))
    for name, st in stats.items():
        assert grad_within_tolerance(st), (name, st)


def test_bwd_scale_argument(fa):
    """A scale other than 1/sqrt(d) is used in both S and the dQ, dK products."""
    q, k, v = make_qkv_gqa(1, 2, 2, 200, 200, 64, seed=4401)
    do = make_dout(q.shape, seed=4402)
    stats = check(q, k, v, do, run(fa, q, k, v, do, True, scale=0.05), 0.05, True)
    print(case_stats_line(stats))
    for name, st in stats.items():
        assert grad_within_tolerance(st), (name, st)


def test_bwd_zero_upstream_gradient(fa):
    """dO = 0 gives exactly zero gradients and D = 0."""
    q, k, v = make_qkv_gqa(1, 2, 1, 300, 300, 128, seed=4501)
    do = torch.zeros_like(q)
    dq, dk, dv, delta = run(fa, q, k, v, do, True)
    for t in (dq, dk, dv, delta):
        assert bool((t == 0).all())


BWD_WORKLOADS = [n for n, w in WORKLOADS.items() if w.direction == "bwd"]


@pytest.mark.parametrize("name", BWD_WORKLOADS)
def test_bwd_workload_full_size_sampled(fa, name):
    """The bench's backward launches (B=2, H=16, causal, N=8192 or 2048) on their own
    inputs; two heads checked in full."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    do = make_workload_dout(w)
    res = run(fa, q, k, v, do, w.causal)
    stats = check(q, k, v, do, res, w.scale, w.causal, kv_heads=[(0, 3), (1, 14)])
    print(case_stats_line(stats))
    for name, st in stats.items():
        assert grad_within_tolerance(st), (name, st)
    assert fa.fa_status(clear=False) == 0


def test_bwd_repeatable_and_status_clean(fa):
    q, k, v = make_qkv_gqa(1, 4, 2, 500, 500, 128, seed=4601)
    do = make_dout(q.shape, seed=4602)
    a = run(fa, q, k, v, do, True)
    b = run(fa, q, k, v, do, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert fa.fa_status(clear=False) == 0


def test_bwd_next_work_on_the_stream_sees_complete_gradients(fa):
    """The dQ kernel is launched as a programmatic dependent of the dK/dV kernel and may start
    before that kernel ends; whatever the stream runs next must still see dQ, dK and dV complete.
    The outputs are filled with NaN, the backward runs, and the next kernels on the same stream
    (copies, with no synchronisation in between) must read exactly a synchronised run's
    gradients."""
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv_gqa(2, 16, 16, 4096, 4096, 128, seed=4801))
    do = make_dout(q.shape, seed=4802).to(dev)
    o, lse = fa.fa_fwd_gqa(q, k, v, causal=True)
    ref = fa.fa_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    ref = [t.clone() for t in ref[:3]]
    for _ in range(3):
        outs = [torch.full_like(t, float("nan")) for t in ref]
        fa.fa_bwd(q, k, v, o, lse, do, dq=outs[0], dk=outs[1], dv=outs[2], causal=True)
        snap = [t.clone() for t in outs]  # the stream's next kernels
        torch.cuda.synchronize()
        for got, want in zip(snap, ref):
            assert torch.equal(got, want)
    assert fa.fa_status(clear=False) == 0


def test_bwd_argument_errors_on_device(fa):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv_gqa(1, 2, 2, 128, 128, 64, seed=4701))
    o, lse = fa.fa_fwd_gqa(q, k, v)
    do = torch.randn_like(q)
    dq = torch.full_like(q, 7.0)
    with pytest.raises(fa.FAError):
        fa.fa_bwd(q, k, v, o, lse, do, dq=q)             # dQ aliases Q
    with pytest.raises(fa.FAError):
        fa.fa_bwd(q, k, v, o, lse, do, dq=dq, dk=do)     # dK aliases dO
    with pytest.raises(fa.FAError):
        fa.fa_bwd(q.cpu(), k, v, o, lse, do, dq=dq, stream=torch.cuda.current_stream())  # host pointer
    torch.cuda.synchronize()
    assert bool((dq == 7.0).all())
