"""Seeded synthetic inputs for the attention forward.

This module holds no attention arithmetic: it only draws random tensors, so
both the CUDA path and the CPU oracle can be fed the same bits.  Q, K and V
are drawn in that order from one ``torch.Generator`` as float32 normals times
a standard deviation, then rounded to bf16 (round-to-nearest-even); the bf16
values convert to float64 exactly on the oracle side.

The workloads are the shapes the attention forward and backward are measured
and checked on; each is named by what it is.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """B batches; H query heads of N rows each; Hkv key/value heads of Nk rows each
    (defaults: Hkv = H, Nk = N); d the head dimension; n_splits key ranges."""
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qk_std: float = 1.0
    v_std: float = 1.0
    seed: int = 0
    Hkv: int | None = None
    Nk: int | None = None
    n_splits: int = 1
    bound: str = "tensor"   # the roofline that bounds it: "tensor" or "hbm"
    direction: str = "fwd"  # "fwd": O and LSE; "bwd": dQ, dK, dV from O, LSE and dO;
                            # "fp8": O and LSE with E4M3 products (fa_fwd_fp8)

    @property
    def hkv(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    @property
    def nk(self) -> int:
        return self.N if self.Nk is None else self.Nk

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def flops(self) -> float:
        """Forward: 4*B*H*Nq*Nk*d (two products, QK^T and PV, of 2*Nq*Nk*d each).
        Backward: 10*B*H*Nq*Nk*d (five products: dV, dP, dQ, dK and the recomputed
        QK^T).  The square causal case counts half."""
        per_pair = 10.0 if self.direction == "bwd" else 4.0
        f = per_pair * self.B * self.H * self.N * self.nk * self.d
        return f / 2.0 if (self.causal and self.N == self.nk) else f

    def algorithmic_bytes(self) -> int:
        """Forward: Q, K, V read once and O written once (bf16), LSE written once (fp32).
        Backward: Q, K, V, O, dO read and dQ, dK, dV written once (bf16), LSE read and
        D written once (fp32)."""
        q_rows = self.B * self.H * self.N
        kv_rows = self.B * self.hkv * self.nk
        if self.direction == "bwd":
            return (4 * q_rows + 4 * kv_rows) * self.d * 2 + 2 * q_rows * 4
        return (2 * q_rows + 2 * kv_rows) * self.d * 2 + q_rows * 4


WORKLOADS = {
    w.name: w
    for w in (
        Workload("n128_d64", 1, 1, 128, 64, False, seed=20261),
        Workload("n2048_d64", 4, 16, 2048, 64, False, seed=20262),
        Workload("causal_n8192_d128", 2, 16, 8192, 128, True, seed=20263),
        Workload("wide_scores_n1024_d128", 8, 32, 1024, 128, False, qk_std=3.0, seed=20264),
        Workload("causal_n32768_d128", 1, 32, 32768, 128, True, seed=20265),
        # grouped K/V heads (8 query heads per K/V head), causal prefill
        Workload("gqa_causal_n8192_d128", 1, 32, 8192, 128, True, seed=20266, Hkv=4),
        # decoding: one new query per head against a 32K-key cache, 4 query heads
        # per K/V head (memory-bound: reads K and V once); the keys are split 4 ways, which
        # the decode kernel runs as 64 groups x 2 CTAs of two splits each (one wave)
        Workload("gqa_decode_nk32768_d128", 8, 32, 1, 128, False, seed=20267, Hkv=8,
                 Nk=32768, n_splits=4, bound="hbm"),
        # the backward of the causal prefill shape: dQ, dK, dV with recomputation
        Workload("bwd_causal_n8192_d128", 2, 16, 8192, 128, True, seed=20263, direction="bwd"),
        # a small backward (inputs of 16 MiB per tensor) for full-section profiler captures
        Workload("bwd_causal_n2048_d128", 2, 16, 2048, 128, True, seed=20268, direction="bwd"),
        # the causal prefill shape through the FP8 path (same inputs as the bf16 headline)
        Workload("fp8_causal_n8192_d128", 2, 16, 8192, 128, True, seed=20263, direction="fp8"),
        Workload("fp8_causal_n2048_d128", 2, 16, 2048, 128, True, seed=20268, direction="fp8"),
    )
}

HEADLINE = "causal_n8192_d128"


def make_qkv(B: int, H: int, N: int, d: int, seed: int, qk_std: float = 1.0,
             v_std: float = 1.0):
    """Return CPU bf16 tensors q, k, v of shape [B, H, N, d] (contiguous)."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, N, d)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    k = (torch.randn(shape, generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    v = (torch.randn(shape, generator=g, dtype=torch.float32) * v_std).to(torch.bfloat16)
    return q, k, v


def make_qkv_gqa(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, seed: int,
                 qk_std: float = 1.0, v_std: float = 1.0):
    """q [B, Hq, Nq, d], k and v [B, Hkv, Nk, d]: CPU bf16, drawn in that order."""
    g = torch.Generator().manual_seed(int(seed))
    q = (torch.randn((B, Hq, Nq, d), generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    k = (torch.randn((B, Hkv, Nk, d), generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    v = (torch.randn((B, Hkv, Nk, d), generator=g, dtype=torch.float32) * v_std).to(torch.bfloat16)
    return q, k, v


def make_dout(shape, seed: int, std: float = 1.0):
    """The upstream gradient dO for the backward: CPU bf16 normals times ``std``,
    drawn from its own Generator(seed)."""
    g = torch.Generator().manual_seed(int(seed))
    return (torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def make_signs(d: int, seed: int):
    """The incoherent-processing rotation's random signs: CPU int8 [d] of +1 / -1 drawn
    from Generator(seed)."""
    g = torch.Generator().manual_seed(int(seed))
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.int8)


def make_workload_signs(w: Workload):
    """The rotation signs of an FP8 workload: seed = the workload's seed + 200."""
    return make_signs(w.d, w.seed + 200)


def make_workload_dout(w: Workload):
    """dO of a backward workload: [B, H, N, d], seed = the workload's seed + 100."""
    return make_dout((w.B, w.H, w.N, w.d), seed=w.seed + 100)


def make_workload(w: Workload):
    if w.Hkv is None and w.Nk is None:
        return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.qk_std, w.v_std)
    return make_qkv_gqa(w.B, w.H, w.hkv, w.N, w.nk, w.d, w.seed, w.qk_std, w.v_std)


def sample_slices(B: int, H: int, count: int, seed: int):
    """``count`` distinct (b, h) pairs drawn from Generator(seed)."""
    g = torch.Generator().manual_seed(int(seed))
    total = B * H
    count = min(count, total)
    idx = torch.randperm(total, generator=g)[:count].tolist()
    return [(i // H, i % H) for i in sorted(idx)]


def sample_rows(N: int, count: int, seed: int, leading: int = 0):
    """``count`` distinct query rows of a length-N sequence: the first ``leading`` rows,
    row 0, the last row and the first/last row of the last 128-row tile, and the rest
    drawn from Generator(seed)."""
    g = torch.Generator().manual_seed(int(seed))
    fixed = set(range(min(leading, N))) | {0, N - 1, max(0, (N - 1) // 128 * 128)}
    perm = torch.randperm(N, generator=g).tolist()
    rest = [r for r in perm if r not in fixed][:max(0, count - len(fixed))]
    return sorted(fixed | set(rest))
