"""GPU tests of fa_fwd_host and fa_bwd_host: the forward and the backward from pinned host
buffers to pinned host buffers, with the copies of one chunk of K/V groups overlapped with the
kernels of another.

Each chunk runs the device entry's kernels on its groups, so the results must equal
fa_fwd_gqa's (fa_bwd's) bit for bit, whatever the chunking; one forward case is also checked
against the fp64 oracle."""
import math

import pytest
import torch

import oracle
from exact_io_aware_02_gb300.inputs import make_qkv_gqa
from tests.parity import compare, within_tolerance

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


def host_run(fa, q, k, v, causal, groups_per_chunk, stream=None):
    """q, k, v: CPU bf16.  Returns (o, lse) on the host, after a synchronise."""
    dev = torch.device("cuda")
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    B, Hq, Nq, d = q.shape
    oh = torch.full(q.shape, 7.0, dtype=torch.bfloat16).pin_memory()
    lh = torch.full((B, Hq, Nq), 7.0, dtype=torch.float32).pin_memory()
    qd, kd, vd = (torch.zeros(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v))
    od = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ld = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, causal=causal, groups_per_chunk=groups_per_chunk,
                   stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    return oh, lh


CASES = [  # B, Hq, Hkv, Nq, Nk, d, causal
    (2, 8, 8, 1000, 1000, 128, True),   # MHA, ragged, causal
    (1, 8, 2, 300, 300, 64, False),     # GQA, d = 64
    (3, 6, 3, 129, 513, 128, True),     # fewer queries than keys, bottom-right mask
    (1, 1, 1, 1, 1, 128, False),        # one group, one row
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}Nq{}Nk{}d{}{}".format(*c[:6], "c" if c[6] else "n"))
@pytest.mark.parametrize("groups_per_chunk", [0, 1, 3, 1000])
def test_host_equals_device_call(fa, case, groups_per_chunk):
    B, Hq, Hkv, Nq, Nk, d, causal = case
    q, k, v = make_qkv_gqa(B, Hq, Hkv, Nq, Nk, d, seed=9100 + Nq + d)
    oh, lh = host_run(fa, q, k, v, causal, groups_per_chunk)
    dev = torch.device("cuda")
    od, ld = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal, n_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())
    assert fa.fa_status(clear=False) == 0


def test_host_matches_oracle(fa):
    B, H, N, d = 2, 4, 700, 128
    q, k, v = make_qkv_gqa(B, H, H, N, N, d, seed=9200)
    oh, lh = host_run(fa, q, k, v, True, 2)
    scale = 1.0 / math.sqrt(d)
    for b in range(B):
        for h in range(H):
            ro, rl = oracle.naive_attention(q[b, h].double().numpy(), k[b, h].double().numpy(),
                                            v[b, h].double().numpy(), scale, True)
            st = compare(oh[b, h].double().numpy(), lh[b, h].double().numpy(), ro, rl)
            assert within_tolerance(st), st


def test_host_on_a_side_stream(fa):
    """The call orders itself after the caller's stream and that stream waits for it."""
    q, k, v = make_qkv_gqa(1, 4, 4, 640, 640, 128, seed=9300)
    s = torch.cuda.Stream()
    oh, lh = host_run(fa, q, k, v, False, 1, stream=s)
    dev = torch.device("cuda")
    od, ld = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())


def test_host_argument_errors(fa):
    dev = torch.device("cuda")
    q, k, v = make_qkv_gqa(1, 2, 2, 256, 256, 128, seed=9400)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((1, 2, 256), dtype=torch.float32).pin_memory()
    qd, kd, vd, od = (torch.empty(q.shape, dtype=torch.bfloat16, device=dev) for _ in range(4))
    ld = torch.empty((1, 2, 256), dtype=torch.float32, device=dev)
    with pytest.raises(fa.FAError):  # pageable host input
        fa.fa_fwd_host(q, kh, vh, oh, lh, qd, kd, vd, od, ld)
    with pytest.raises(fa.FAError):  # pageable host output
        fa.fa_fwd_host(qh, kh, vh, torch.empty_like(q), lh, qd, kd, vd, od, ld)
    with pytest.raises(fa.FAError):  # host output over a host input
        fa.fa_fwd_host(qh, kh, vh, qh, lh, qd, kd, vd, od, ld)
    with pytest.raises(fa.FAError):  # negative chunk size
        fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, groups_per_chunk=-1)
    with pytest.raises(fa.FAError):  # device output over a device input
        fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, qd, ld)
    torch.cuda.synchronize()


BWD_CASES = [  # B, Hq, Hkv, N, d, causal
    (2, 4, 4, 1000, 128, True),   # ragged, causal
    (1, 8, 2, 300, 64, False),    # grouped K/V heads, d = 64
    (3, 2, 1, 77, 128, True),     # tiny ragged rows per group
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "B{}Hq{}Hkv{}N{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
@pytest.mark.parametrize("groups_per_chunk", [0, 1, 1000])
def test_bwd_host_equals_device_call(fa, case, groups_per_chunk):
    from exact_io_aware_02_gb300.inputs import make_dout
    B, Hq, Hkv, N, d, causal = case
    dev = torch.device("cuda")
    q, k, v = make_qkv_gqa(B, Hq, Hkv, N, N, d, seed=9500 + N + d)
    do = make_dout(q.shape, seed=9600 + N)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_gqa(qd, kd, vd, causal=causal)
    ref = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    hin = tuple(t.cpu().contiguous().pin_memory() for t in (q, k, v, o, lse, do))
    hout = tuple(torch.full(t.shape, 7.0, dtype=t.dtype).pin_memory() for t in (q, k, v))
    din = tuple(torch.zeros_like(t) for t in (qd, kd, vd, o, lse, dod))
    dout_ = tuple(torch.empty_like(t) for t in (qd, kd, vd))
    delta = torch.empty_like(lse)
    fa.fa_bwd_host(hin, hout, din, dout_, delta, causal=causal, groups_per_chunk=groups_per_chunk)
    torch.cuda.synchronize()
    for got, want in zip(hout, ref[:3]):
        assert torch.equal(got, want.cpu())
    assert torch.equal(delta, ref[3])
    assert fa.fa_status(clear=False) == 0


def test_bwd_host_argument_errors(fa):
    from exact_io_aware_02_gb300.inputs import make_dout
    dev = torch.device("cuda")
    q, k, v = make_qkv_gqa(1, 2, 2, 256, 256, 128, seed=9700)
    do = make_dout(q.shape, seed=9701)
    lse = torch.zeros((1, 2, 256), dtype=torch.float32)
    hin = tuple(t.pin_memory() for t in (q, k, v, q.clone(), lse, do))
    hout = tuple(torch.empty_like(t).pin_memory() for t in (q, k, v))
    din = tuple(t.to(dev) for t in (q, k, v, q, lse, do))
    dout_ = tuple(torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v))
    delta = torch.empty((1, 2, 256), dtype=torch.float32, device=dev)
    with pytest.raises(fa.FAError):  # pageable host input
        fa.fa_bwd_host((q,) + hin[1:], hout, din, dout_, delta)
    with pytest.raises(fa.FAError):  # host output over a host input
        fa.fa_bwd_host(hin, (hin[0],) + hout[1:], din, dout_, delta)
    with pytest.raises(fa.FAError):  # negative chunk size
        fa.fa_bwd_host(hin, hout, din, dout_, delta, groups_per_chunk=-1)
    torch.cuda.synchronize()


def test_host_calls_from_two_threads(fa):
    """Two host threads call fa_fwd_host at once on their own streams: the library enqueues
    whole calls one at a time (its events are shared), and both results are exact."""
    import threading
    dev = torch.device("cuda")
    probs = [make_qkv_gqa(1, 6, 6, 640, 640, 128, seed=9800 + i) for i in range(2)]
    want = []
    for q, k, v in probs:
        o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
        want.append((o.cpu(), lse.cpu()))
    torch.cuda.synchronize()
    got = [None, None]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            for _ in range(3):
                got[i] = host_run(fa, *probs[i], True, 2, stream=s)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)
    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (oh, lh), (o, lse) in zip(got, want):
        assert torch.equal(oh, o) and torch.equal(lh, lse)
