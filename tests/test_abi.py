"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks that run before any CUDA call (no GPU)."""
import ctypes
import os
import re

import pytest

import __graft_entry__ as entry

HEADER = os.path.join(entry.ROOT, "include", "fa_gb300.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def fa():
    entry.build()
    from exact_io_aware_02_gb300 import fa as mod
    return mod


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "fa_fwd" in names and "fa_strerror" in names and "fa_status" in names


def test_library_exports_every_declared_symbol(fa):
    for name in declared_functions():
        assert hasattr(fa.lib, name), name
        assert isinstance(getattr(fa.lib, name), ctypes._CFuncPtr)
    assert set(fa.EXPORTED) == set(declared_functions())


def test_strerror_and_version(fa):
    assert fa.fa_version() == 3
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert fa.fa_strerror(code) and fa.fa_strerror(code) != "unknown error"
    assert fa.fa_strerror(-99) == "unknown error"


FAKE = 0x7f0000000000  # 16-byte aligned, never dereferenced: rejected before any CUDA call


def _call(fa, q=FAKE, k=FAKE + 2**30, v=FAKE + 2**31, o=FAKE + 3 * 2**30, lse=FAKE + 2**32,
          B=1, H=1, N=128, d=128, scale=0.088, causal=0):
    return fa.lib.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


@pytest.mark.parametrize("kw", [
    {"q": 0}, {"k": 0}, {"v": 0}, {"o": 0}, {"lse": 0},
    {"d": 96}, {"d": 256}, {"d": 0}, {"B": 0}, {"H": -1}, {"N": 0},
    {"scale": 0.0}, {"scale": -1.0}, {"scale": float("inf")}, {"scale": float("nan")},
    {"q": FAKE + 8}, {"o": FAKE + 3 * 2**30 + 4}, {"lse": FAKE + 2**32 + 4},
    {"B": 65536, "H": 65536, "N": 2},
    {"o": FAKE},                       # output overlaps an input
    {"lse": FAKE + 3 * 2**30 + 64},    # LSE overlaps O
])
def test_argument_errors_before_launch(fa, kw):
    assert _call(fa, **kw) == fa.FA_ERR_ARG


def test_fp8_sequence_limit(fa):
    """The FP8 forward keeps per-tile tables of at most 1024 key tiles: N = 131072 is the
    largest length it accepts; one more row is rejected before any CUDA call."""
    ws = fa.lib.fa_fwd_fp8_workspace_bytes
    assert ws(1, 1, 131072, 128) > 0
    args = [FAKE + i * 2**30 for i in range(6)]
    assert fa.lib.fa_fwd_fp8(*args, 1, 1, 131073, 128, 0.088, 0, FAKE + 7 * 2**30, 1 << 40, None) == fa.FA_ERR_ARG


def test_bwd_and_fp8_withheld_timeout_range(fa):
    b = fa.lib.fa_bwd_withheld_tile
    args = [FAKE + i * 2**30 for i in range(10)] + [1, 2, 1, 128, 128, 0.088, 1]
    assert b(*args, 0.5, None) == fa.FA_ERR_ARG
    assert b(*args, 20000.0, None) == fa.FA_ERR_ARG
    f8 = fa.lib.fa_fwd_fp8_withheld_tile
    args8 = [FAKE + i * 2**30 for i in range(6)] + [1, 1, 128, 128, 0.088, 0, FAKE + 7 * 2**30, 1 << 20]
    assert f8(*args8, 0.0, None) == fa.FA_ERR_ARG
    assert f8(*args8, 1e9, None) == fa.FA_ERR_ARG


def test_withheld_tile_timeout_range(fa):
    f = fa.lib.fa_fwd_withheld_tile
    assert f(FAKE, FAKE + 2**30, FAKE + 2**31, FAKE + 3 * 2**30, FAKE + 2**32, 1, 1, 128, 128,
             0.088, 0, 0.5, None) == fa.FA_ERR_ARG
    assert f(FAKE, FAKE + 2**30, FAKE + 2**31, FAKE + 3 * 2**30, FAKE + 2**32, 1, 1, 128, 128,
             0.088, 0, 20000.0, None) == fa.FA_ERR_ARG


def test_withheld_ring_tile_arguments(fa):
    f = fa.lib.fa_fwd_withheld_ring_tile
    ptrs = (FAKE, FAKE + 2**30, FAKE + 2**31, FAKE + 3 * 2**30, FAKE + 2**32)
    assert f(*ptrs, 1, 1, 128, 128, 0.088, 0, -1, 50.0, None) == fa.FA_ERR_ARG  # no tile named
    assert f(*ptrs, 1, 1, 128, 128, 0.088, 0, 3, 0.5, None) == fa.FA_ERR_ARG
    assert f(*ptrs, 1, 1, 128, 128, 0.088, 0, 3, 20000.0, None) == fa.FA_ERR_ARG


def _bwd(fa, B=1, Hq=2, Hkv=1, N=128, d=128, scale=0.088, causal=1, **ptrs):
    names = ("q", "k", "v", "o", "lse", "dout", "dq", "dk", "dv", "delta")
    p = {n: FAKE + i * 2**30 for i, n in enumerate(names)}
    p.update(ptrs)
    return fa.lib.fa_bwd(*(p[n] for n in names), B, Hq, Hkv, N, d, scale, causal, None)


@pytest.mark.parametrize("kw", [
    {"q": 0}, {"lse": 0}, {"dout": 0}, {"dq": 0}, {"dk": 0}, {"dv": 0}, {"delta": 0},
    {"d": 96}, {"d": 32}, {"B": 0}, {"N": 0}, {"Hq": 3, "Hkv": 2}, {"Hkv": 0},
    {"scale": 0.0}, {"scale": float("nan")},
    {"dq": FAKE + 6 * 2**30 + 8}, {"delta": FAKE + 9 * 2**30 + 4},
    {"dq": FAKE},                       # dQ overlaps Q
    {"dk": FAKE + 6 * 2**30 + 256},     # dK overlaps dQ
    {"delta": FAKE + 4 * 2**30},        # D overlaps LSE
    {"B": 65536, "Hq": 65536, "Hkv": 65536, "N": 2},
])
def test_bwd_argument_errors_before_launch(fa, kw):
    assert _bwd(fa, **kw) == fa.FA_ERR_ARG


def test_host_entry_argument_errors(fa):
    f = fa.lib.fa_fwd_host
    dev = [FAKE + i * 2**30 for i in range(5)]
    host = [FAKE + (8 + i) * 2**30 for i in range(5)]
    tail = [1, 2, 2, 128, 128, 128, 0.088, 0]
    assert f(*([0] + host[1:]), *dev, *tail, 0, None) == fa.FA_ERR_ARG  # null host input
    assert f(*host, *dev, *tail, -1, None) == fa.FA_ERR_ARG              # negative chunk size
    assert f(*host, *dev, 1, 2, 2, 128, 128, 96, 0.088, 0, 0, None) == fa.FA_ERR_ARG  # d = 96


def test_bwd_host_entry_argument_errors(fa):
    f = fa.lib.fa_bwd_host
    host = [FAKE + (20 + i) * 2**30 for i in range(9)]
    dev = [FAKE + i * 2**30 for i in range(10)]
    tail = [1, 2, 2, 128, 128, 0.088, 0]
    assert f(*([0] + host[1:]), *dev, *tail, 0, None) == fa.FA_ERR_ARG  # null host input
    assert f(*host, *dev, *tail, -1, None) == fa.FA_ERR_ARG              # negative chunk size



def _gqa_pair(fa, **kw):
    """fa_fwd_gqa (with a fake workspace of the size it asks for) and
    fa_fwd_gqa_static_workspace on the same arguments."""
    a = dict(q=FAKE, k=FAKE + 2**30, v=FAKE + 2**31, o=FAKE + 3 * 2**30, lse=FAKE + 2**32,
             B=1, Hq=4, Hkv=2, Nq=1, Nk=512, d=128, scale=0.088, causal=0, n_splits=4)
    a.update(kw)
    ptrs = [a[n] for n in ("q", "k", "v", "o", "lse")]
    sizes = [a[n] for n in ("B", "Hq", "Hkv", "Nq", "Nk", "d")]
    need = fa.lib.fa_fwd_gqa_workspace_bytes(a["B"], a["Hq"], a["Nq"], a["d"], a["n_splits"])
    rc_gqa = fa.lib.fa_fwd_gqa(*ptrs, *sizes, a["scale"], a["causal"], a["n_splits"],
                               FAKE + 5 * 2**30, need, None)
    rc_static = fa.lib.fa_fwd_gqa_static_workspace(*ptrs, *sizes, a["scale"], a["causal"], a["n_splits"], None)
    return rc_gqa, rc_static


@pytest.mark.parametrize("kw", [
    {"q": 0}, {"lse": 0}, {"d": 96}, {"Hkv": 3}, {"Nk": 0}, {"scale": 0.0}, {"q": FAKE + 8},
    {"o": FAKE},            # output overlaps an input
    {},                     # well-formed, but not device memory (fake addresses)
])
def test_static_workspace_entry_reports_like_fa_fwd_gqa(fa, kw):
    """The no-allocation entry point checks its arguments as fa_fwd_gqa does, before it
    touches the device, so both return the same code (here all are argument errors: the
    addresses are fake)."""
    rc_gqa, rc_static = _gqa_pair(fa, **kw)
    assert rc_static == rc_gqa == fa.FA_ERR_ARG, (rc_gqa, rc_static)


def test_static_workspace_entry_rejects_oversized_before_any_device_call(fa):
    need = fa.lib.fa_fwd_gqa_workspace_bytes(1, 64, 64, 128, 16)
    assert need > fa.FA_STATIC_WORKSPACE_BYTES
    _, rc_static = _gqa_pair(fa, Hq=64, Hkv=8, Nq=64, n_splits=16)
    assert rc_static == fa.FA_ERR_WORKSPACE_TOO_LARGE
