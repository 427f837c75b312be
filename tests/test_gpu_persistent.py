"""GPU parity of the forward when each persistent CTA runs many work items in a row.

A work item is a pair of 128-row query tiles of one group over one K/V split; the grid holds
one CTA per item and a running CTA takes over CTAs that have not started yet.  Most parity
cases have fewer items than the GPU has SMs, so each CTA runs one item.  These shapes have
hundreds of items, so CTAs carry the K/V ring, the barrier phases, the V scale and the O
staging slots from item to item, across the cases that change an item's shape: a pair with one
tile (an odd number of query tiles), items whose rows see no key at all (more queries than keys,
causal), K/V splits written as partials and merged, and d = 64.  Sampled heads and rows of each
are compared with the fp64 oracle, and the status word must stay clean."""
import math

import pytest
import torch

import oracle
from exact_io_aware_02_gb300.inputs import make_qkv_gqa
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


CASES = [  # B, Hq, Hkv, Nq, Nk, d, causal, n_splits; items = B * Hkv * ceil(ceil(Hq/Hkv*Nq/128)/2) * splits
    (1, 160, 160, 384, 384, 128, False, 1),   # 320 items, every second one a single tile
    (1, 96, 96, 640, 640, 64, True, 1),       # 288 items of 1 to 5 K/V steps
    (4, 32, 8, 1024, 512, 128, True, 1),      # 512 items, rows 0-511 of every head see no key
    (1, 40, 40, 2048, 2048, 128, False, 2),   # 640 items over two K/V splits, merged
    (2, 64, 16, 384, 1000, 64, True, 1),      # 192 items, query tiles straddling heads, ragged keys
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,n_splits", CASES,
                         ids=[f"B{a}Hq{b}Hkv{c}Nq{e}Nk{f}d{g}{'c' if h else 'n'}s{i}" for a, b, c, e, f, g, h, i in CASES])
def test_many_items_per_cta(fa, B, Hq, Hkv, Nq, Nk, d, causal, n_splits):
    q, k, v = make_qkv_gqa(B, Hq, Hkv, Nq, Nk, d, seed=5100 + Hq + Nq + Nk + d)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda")
    fa.fa_status(clear=True)
    o, lse = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal, n_splits=n_splits)
    torch.cuda.synchronize()
    assert fa.fa_status(clear=True) == 0
    o, lse = o.cpu(), lse.cpu()
    G = Hq // Hkv
    # the first, middle and last heads of the first and last batch entries
    heads = sorted({(0, 0), (0, 1), (0, Hq // 2), (B - 1, Hq - 2), (B - 1, Hq - 1)})
    rows = sorted({0, 1, 127, 128, 255, 256, Nq // 2, Nq - 129, Nq - 128, Nq - 1} | set(range(0, Nq, 53)))
    rows = [r for r in rows if 0 <= r < Nq]
    stats = []
    for b, h in heads:
        ro, rl = oracle.naive_attention(_np64(q[b, h]), _np64(k[b, h // G]), _np64(v[b, h // G]),
                                        scale, causal, rows=rows, q_offset=Nk - Nq)
        stats.append(compare(_np64(o[b, h][rows]), _np64(lse[b, h][rows]), ro, rl))
    st = merge(stats)
    log_stats(f"persistent_B{B}Hq{Hq}Hkv{Hkv}Nq{Nq}Nk{Nk}d{d}{'c' if causal else 'n'}s{n_splits}", st, heads, len(rows))
    assert within_tolerance(st), st
    # every element finite, and rows that see no key at all: O = 0, LSE = -inf
    assert torch.isfinite(o.float()).all()
    if causal and Nq > Nk:
        blind = Nq - Nk  # rows 0 .. Nq - Nk - 1 of every head
        assert torch.all(o[:, :, :blind].float() == 0)
        assert torch.all(torch.isneginf(lse[:, :, :blind]))
