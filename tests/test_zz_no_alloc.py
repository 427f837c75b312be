"""fa_fwd_gqa_static_workspace: the entry point for callers that cannot allocate
device memory (a serving loop with a fixed memory plan, a plain C host without an
allocator).  It must give the same results as fa_fwd_gqa with a caller workspace,
call after call, although every call reuses the library's one fixed array.

This file is collected last on purpose, and it also passes on its own in a fresh
process."""
import ctypes
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
    return mod


def _np64(t):
    return t.to(torch.float64).cpu().numpy()


def _static_call(fa, q, k, v, o, lse, causal, n_splits, stream):
    """Straight through the C ABI; the outputs are preallocated, nothing else is."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    return fa.lib.fa_fwd_gqa_static_workspace(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, Hq, Hkv, Nq, Nk, d,
        ctypes.c_float(1.0 / math.sqrt(d)), int(causal), n_splits, ctypes.c_void_p(stream))


CASES = [  # B, Hq, Hkv, Nq, Nk, d, causal, n_splits
    (4, 32, 8, 1, 8192, 128, False, 16),   # decoding against a long cache
    (2, 8, 2, 5, 3000, 64, True, 7),       # a few new queries, bottom-right causal
]


@pytest.mark.parametrize("case", CASES, ids=["decode_d128", "few_queries_d64"])
def test_static_workspace_matches_caller_workspace_twice(fa, case):
    """Same kernels, same inputs: the results must be bit-identical to fa_fwd_gqa's with a
    caller workspace, on each of two calls in a row (a stale partial left in the shared
    array by the first call would show up in the second).  One query head per call is
    also checked against the oracle directly."""
    B, Hq, Hkv, Nq, Nk, d, causal, n_splits = case
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((901, 902)):  # two calls in a row, different inputs
        qc, kc, vc = make_qkv_gqa(B, Hq, Hkv, Nq, Nk, d, seed=seed + d)
        q, k, v = (t.to(dev) for t in (qc, kc, vc))
        o_ref, lse_ref = fa.fa_fwd_gqa(q, k, v, causal=causal, n_splits=n_splits)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, Nq), float("nan"), device=dev)
        assert _static_call(fa, q, k, v, o, lse, causal, n_splits, stream) == fa.FA_OK
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), call
        assert torch.equal(lse, lse_ref), call
        b, h = B - 1, Hq - 1 - call
        G = Hq // Hkv
        ro, rl = oracle.naive_attention(qc[b, h].double().numpy(), kc[b, h // G].double().numpy(),
                                        vc[b, h // G].double().numpy(), 1.0 / math.sqrt(d), causal,
                                        q_offset=Nk - Nq)
        st = compare(_np64(o[b, h]), _np64(lse[b, h]), ro, rl)
        assert within_tolerance(st), (call, st)


def test_static_workspace_rejects_oversized_splits(fa):
    dev = torch.device("cuda")
    B, Hq, Nq, d, n_splits = 1, 64, 64, 128, 16          # needs more than the fixed 16 MiB
    assert fa.fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits) > fa.FA_STATIC_WORKSPACE_BYTES
    q, k, v = (t.to(dev) for t in make_qkv_gqa(B, Hq, 8, Nq, 256, d, seed=903))
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, Hq, Nq), 3.0, device=dev)
    rc = _static_call(fa, q, k, v, o, lse, False, n_splits, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_ERR_WORKSPACE_TOO_LARGE
    torch.cuda.synchronize()
    assert bool((o == 3.0).all()) and bool((lse == 3.0).all())   # nothing was enqueued
    assert fa.fa_status(clear=False) == 0
