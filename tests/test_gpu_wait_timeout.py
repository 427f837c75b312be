"""Bounded device waits: a kernel whose producer never loads one V tile gives up
after the short wait limit, raises the status bit, frees its resources and
returns; the context stays usable (no fault, no hang)."""
import math

import pytest
import torch

from exact_io_aware_02_gb300.inputs import make_dout, make_qkv, make_qkv_gqa, make_signs

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_cleanly():
    import __graft_entry__ as entry
    entry.build()
    from exact_io_aware_02_gb300 import fa

    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 512, 128, seed=21))
    fa.fa_status(clear=True)
    rc = fa.fa_fwd_withheld_tile(q, k, v, wait_timeout_ms=50.0)
    assert rc == fa.FA_OK
    status = fa.fa_status(clear=True)
    assert status & fa.FA_STATUS_TIMEOUT
    # the context still works and a normal call leaves the status clean
    o, lse = fa.fa_fwd(q, k, v, scale=1 / math.sqrt(128), causal=False)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert fa.fa_status(clear=False) == 0


@pytest.mark.parametrize("ring_tile", [2, 5, 6])
@pytest.mark.parametrize("causal", [False, True])
def test_withheld_later_tile_times_out_cleanly(ring_tile, causal):
    """A missing K or V tile after some K/V steps have completed: the softmax warps have handed
    P over for the earlier steps (the MMA warp waited for them at the named barrier), then the
    waits give up; with causal masking the CTAs with fewer tiles complete normally."""
    import __graft_entry__ as entry
    entry.build()
    from exact_io_aware_02_gb300 import fa

    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 1024, 128, seed=26 + ring_tile))
    fa.fa_status(clear=True)
    assert fa.fa_fwd_withheld_ring_tile(q, k, v, ring_tile, causal=causal, wait_timeout_ms=50.0) == fa.FA_OK
    assert fa.fa_status(clear=True) & fa.FA_STATUS_TIMEOUT
    o, lse = fa.fa_fwd(q, k, v, scale=1 / math.sqrt(128), causal=causal)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert fa.fa_status(clear=False) == 0


def test_backward_withheld_tiles_time_out_cleanly():
    """Both backward kernels: a stage (dK/dV) and a V tile (dQ) that never arrive."""
    import __graft_entry__ as entry
    entry.build()
    from exact_io_aware_02_gb300 import fa

    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv_gqa(1, 4, 2, 384, 384, 128, seed=22))
    do = make_dout(q.shape, seed=23).to(dev)
    o, lse = fa.fa_fwd_gqa(q, k, v, causal=True)
    fa.fa_status(clear=True)
    assert fa.fa_bwd_withheld_tile(q, k, v, o, lse, do, wait_timeout_ms=50.0, causal=True) == fa.FA_OK
    assert fa.fa_status(clear=True) & fa.FA_STATUS_TIMEOUT
    dq, dk, dv, _ = fa.fa_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert all(torch.isfinite(t.float()).all() for t in (dq, dk, dv))
    assert fa.fa_status(clear=False) == 0


def test_fp8_withheld_tile_times_out_cleanly():
    import __graft_entry__ as entry
    entry.build()
    from exact_io_aware_02_gb300 import fa

    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 512, 128, seed=24))
    signs = make_signs(128, 25).to(dev)
    fa.fa_status(clear=True)
    assert fa.fa_fwd_fp8_withheld_tile(q, k, v, signs, wait_timeout_ms=50.0) == fa.FA_OK
    assert fa.fa_status(clear=True) & fa.FA_STATUS_TIMEOUT
    o, lse = fa.fa_fwd_fp8(q, k, v, signs)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert fa.fa_status(clear=False) == 0
