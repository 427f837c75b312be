"""Bounded device waits: a kernel whose producer never loads one V tile gives up
after the short wait limit, raises the status bit, frees its resources and
returns; the context stays usable (no fault, no hang)."""
import math

import pytest
import torch

from exact_io_aware_02_gb300.inputs import make_qkv

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
