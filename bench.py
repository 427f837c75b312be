"""Benchmark of the exact attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one fa_fwd call over the whole workload (every (b, h) and query
tile), inputs resident in HBM.  The default workload is the causal
B=2 H=16 N=8192 d=128 forward; the metric is forward TFLOP/s with
4*B*H*N^2*d flops, halved for causal.  Prints one JSON line (rank 0).

Other workloads (--workload): grouped K/V prefill, split-K/V decoding (reported
as HBM GB/s), and the backward of the causal prefill shape (one step = one
fa_bwd call from the forward's O and LSE; 10*B*H*N^2*d flops, halved for causal).

--impl reference times the fp64 CPU oracle on the host cores instead (each
step: one 128-row query tile of one (b, h) slice of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_io_aware_02_gb300.inputs import (HEADLINE, WORKLOADS, make_workload, make_workload_dout,  # noqa: E402
                                            make_workload_signs)

METRIC = "fwd attention TFLOP/s & % of GB300 bf16 tensor peak (B=2 H=16 N=8K d=128 causal)"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
CSRC = os.path.join(ROOT, "exact_io_aware_02_gb300", "csrc")
KERNEL_FILES = {  # the sources each direction's kernels are built from
    "fwd": [os.path.join(CSRC, f) for f in ("fa_fwd_sm103.cu", "fa_common.cuh", "sm103_ptx.cuh")],
    "bwd": [os.path.join(CSRC, f) for f in ("fa_bwd_sm103.cu", "fa_common.cuh", "sm103_ptx.cuh")],
    "fp8": [os.path.join(CSRC, f) for f in ("fa_fp8_sm103.cu", "fa_common.cuh", "sm103_ptx.cuh")],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def _code_only(text: str) -> str:
    """The source without its comments and with runs of white space collapsed, so that the
    digest changes with the code, not with its wording."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal: copied whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_digest(direction: str = "fwd") -> str:
    """sha256 prefix of the code (comments removed) the direction's kernels are built from."""
    h = hashlib.sha256()
    for f in KERNEL_FILES[direction]:
        h.update(_code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (same digest); else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    digest = kernel_digest(WORKLOADS[workload].direction)
    for line in open(TRAFFIC_FILE, encoding="utf-8"):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == digest:
            return float(parts[2])
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    return 1900.0, 6800.0, "fallback"


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a per-rank number over all ranks (identity on one rank)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, ms: float, world: int) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def job_rate(units_per_rank: float, ms: float, world: int) -> float:
    """Whole-job rate in units per second (units: TFLOP or GB per step)."""
    return world * units_per_rank / (ms * 1e-3)


L2_NOTE = "GPU arm: a 256 MiB buffer is written between timed launches (L2 flushed); CUDA events per launch"


def workload_config(w):
    """The workload's description, the same in both arms (the L2 note says how the GPU arm
    keeps timed launches from reusing L2; the CPU arm has no such cache to flush)."""
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
           "qk_std": w.qk_std, "v_std": w.v_std, "seed": w.seed, "l2": L2_NOTE}
    if w.Hkv is not None or w.Nk is not None:
        cfg.update({"Hkv": w.hkv, "Nk": w.nk, "n_splits": w.n_splits})
    return cfg


def metric_for(w):
    """The headline metric for tensor-bound workloads; HBM bytes per second for the
    memory-bound decoding workload (K and V are read once)."""
    if w.bound == "hbm":
        return f"decode attention GB/s of algorithmic HBM traffic ({w.name})", "GB/s"
    if w.direction == "bwd":
        return f"bwd attention TFLOP/s, 10*N^2*d per head, halved for causal ({w.name})", UNIT
    if w.direction == "fp8":
        return f"fp8 (E4M3) fwd attention TFLOP/s, 4*N^2*d per head, halved for causal ({w.name})", UNIT
    return METRIC if w.name == HEADLINE else f"fwd attention TFLOP/s ({w.name})", UNIT


def units_per_step(w):
    return w.algorithmic_bytes() / 1e9 if w.bound == "hbm" else w.flops() / 1e12


def backward_call(fa, w):
    """One backward step through the public API: fa_bwd from the forward's O and LSE."""
    return lambda q, k, v, o, lse, do, grads, stream: fa.fa_bwd(
        q, k, v, o, lse, do, *grads, scale=w.scale, causal=w.causal, stream=stream)


def forward_call(fa, w):
    """The public-API call that does one step of the workload."""
    if w.Hkv is None and w.Nk is None:
        return lambda q, k, v, o, lse, ws, stream: fa.fa_fwd(q, k, v, o, lse, scale=w.scale, causal=w.causal,
                                                             stream=stream)
    return lambda q, k, v, o, lse, ws, stream: fa.fa_fwd_gqa(q, k, v, o, lse, scale=w.scale, causal=w.causal,
                                                             n_splits=w.n_splits, workspace=ws, stream=stream)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self):
        return time.perf_counter()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.05]
        if not inside and rows:  # region shorter than the sampling period: nearest sample
            inside = [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))]
        sm = [float(p[0]) for _, p in inside if p[0].replace(".", "").isdigit()]
        busy = [float(p[0]) for _, p in inside if p[0].replace(".", "").isdigit()
                and p[3].isdigit() and int(p[3]) > 0]
        mx = [float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit()]
        reasons = sorted({name for _, p in inside for name, val in zip(self.NAMES, p[4:])
                          if val.strip().lower() == "active"})
        use = busy or sm
        return {"sm_mhz": statistics.median(use) if use else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(inside)}


def gpu_selector(dev) -> str:
    """nvidia-smi -i argument for a torch device: its UUID when torch knows it."""
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if uuid is not None:
        text = str(uuid)
        return text if text.startswith("GPU-") else "GPU-" + text
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    if visible:
        return visible.split(",")[dev.index or 0].strip()
    return str(dev.index or 0)


def cpu_baseline(w, results=None, budget_s=12.0, max_slices=32):
    """The fp64 oracle as it stands, on whole (b, h) slices of the workload until
    about ``budget_s`` seconds of CPU work; TFLOP/s counted like the GPU metric.

    With ``results`` (the GPU arm's outputs as CPU tensors: (O, LSE) for a forward,
    (dQ, dK, dV) for the backward) the same oracle slices also give the raw parity
    statistics of those outputs, returned as a second value."""
    import numpy as np
    import oracle
    import oracle.fp8 as oracle_fp8
    from exact_io_aware_02_gb300.inputs import sample_slices
    from tests.parity import compare, grad_compare, grad_within_tolerance, merge, within_tolerance

    q, k, v = make_workload(w)
    do = make_workload_dout(w) if w.direction == "bwd" else None
    signs = make_workload_signs(w).numpy().astype(np.float64) if w.direction == "fp8" else None
    G = w.H // w.hkv
    slices = sample_slices(w.B, w.H, max_slices, w.seed + 3)
    per_slice = units_per_step(w) / (w.B * w.H)
    done, t_total = 0, 0.0
    stats = []
    f64 = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    for (b, h) in slices:
        qa = f64(q[b, h])
        ka, va = (f64(t[b, h // G]) for t in (k, v))
        t0 = time.perf_counter()
        if do is not None:
            ref = oracle.attention_backward(qa, ka, va, f64(do[b, h]), w.scale, w.causal)
        elif signs is not None:
            ref = oracle_fp8.fp8_attention(qa, ka, va, w.scale, w.causal, signs)
        else:
            ref = oracle.naive_attention(qa, ka, va, w.scale, w.causal, q_offset=w.nk - w.N)
        t_total += time.perf_counter() - t0
        done += 1
        if results is not None:
            if do is not None:  # one query head per K/V head in the backward workloads
                stats.append([grad_compare(f64(results[i][b, h]), ref[i]) for i in range(3)])
            else:
                stats.append(compare(f64(results[0][b, h]), f64(results[1][b, h]), ref[0], ref[1]))
        if t_total >= budget_s:
            break
    base = {"value": done * per_slice / t_total, "unit": metric_for(w)[1],
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{done} whole (b,h) query-head slice(s) of {w.name} (N={w.N}, d={w.d}, {w.direction}), "
                      f"fp64 NumPy, "
                      f"{t_total:.1f} s; threads = NumPy BLAS default on the listed cores"}
    if results is None:
        return base, None
    where = f"{done} whole (b,h) slice(s) drawn with seed {w.seed + 3}, every row"
    if do is not None:
        parity = {"against": "oracle.attention_backward (fp64)", "slices": where}
        for i, name in enumerate(("dq", "dk", "dv")):
            parity[name] = {"max_rel": max(s[i]["max_rel"] for s in stats),
                            "mean_rel": max(s[i]["mean_rel"] for s in stats)}
        parity["within_tolerance"] = all(grad_within_tolerance(s[i]) for s in stats for i in range(3))
        return base, parity
    st = merge(stats)
    parity = {"against": ("oracle.fp8.fp8_attention (fp64, exact attention of the dequantised tensors)"
                          if signs is not None else "oracle.naive_attention (fp64)"),
              "slices": where, **{key: st[key] for key in ("max_abs_o", "max_abs_o_below4", "mean_abs_o",
                                                          "max_rel_lse", "count")}}
    if signs is None:
        parity["within_tolerance"] = within_tolerance(st)
    return base, parity


def run_reference(args, w, rank, world):
    """Reference arm: the CPU oracle, rank 0 only.  Each step is one 128-row query
    tile of one query head (its K/V head under grouping), fp64 NumPy."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    import oracle.fp8 as oracle_fp8

    q, k, v = make_workload(w)
    do = make_workload_dout(w) if w.direction == "bwd" else None
    signs = make_workload_signs(w).numpy().astype(np.float64) if w.direction == "fp8" else None
    G = w.H // w.hkv
    q_offset = w.nk - w.N
    n_tiles = (w.N + 127) // 128
    per_pair = 10.0 if do is not None else 4.0
    total_units, total_t = 0.0, 0.0

    def step(s, timed):
        nonlocal total_units, total_t
        idx = (s * 7919) % (w.B * w.H * n_tiles)
        bh, tile = divmod(idx, n_tiles)
        b, h = divmod(bh, w.H)
        rows = list(range(tile * 128, min(w.N, tile * 128 + 128)))
        qa = q[b, h].to(torch.float64).numpy()
        ka, va = (t[b, h // G].to(torch.float64).numpy() for t in (k, v))
        t0 = time.perf_counter()
        if do is not None:  # this tile's rows: dQ, and their share of dK and dV
            oracle.attention_backward(qa[rows[0]:rows[-1] + 1], ka, va,
                                      do[b, h, rows[0]:rows[-1] + 1].to(torch.float64).numpy(),
                                      w.scale, w.causal, q_offset=q_offset + rows[0])
        elif signs is not None:
            oracle_fp8.fp8_attention(qa, ka, va, w.scale, w.causal, signs, rows=rows)
        else:
            oracle.naive_attention(qa, ka, va, w.scale, w.causal, rows=rows, q_offset=q_offset)
        dt = time.perf_counter() - t0
        if timed:
            if w.bound == "hbm":
                total_units += len(rows) / (w.B * w.H * w.N) * w.algorithmic_bytes() / 1e9
            else:
                keys = [min(w.nk, q_offset + i + 1) if w.causal else w.nk for i in rows]
                total_units += sum(per_pair * kk * w.d for kk in keys) / 1e12
            total_t += dt

    for s in range(args.warmup):
        step(s, False)
    for s in range(args.steps):
        step(args.warmup + s, True)
    value = total_units / total_t
    metric, unit = metric_for(w)
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} steps of one 128-row query tile of one query head "
                                       f"each ({w.direction}), fp64 NumPy"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_ours(args, w, rank, world, local_rank):
    from exact_io_aware_02_gb300 import fa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    qh, kh, vh = (t.pin_memory() for t in make_workload(w))
    q, k, v = (t.to(dev, non_blocking=True) for t in (qh, kh, vh))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    ws_bytes = fa.fa_fwd_gqa_workspace_bytes(w.B, w.H, w.N, w.d, w.n_splits)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    fwd = forward_call(fa, w)
    if w.direction == "bwd":
        # the backward's inputs: the forward's O and LSE (computed once, untimed) and dO
        fwd(q, k, v, o, lse, ws, stream)
        doh = make_workload_dout(w).pin_memory()
        do = doh.to(dev, non_blocking=True)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev))
        bwd = backward_call(fa, w)
        step = lambda: bwd(q, k, v, o, lse, do, grads, stream)  # noqa: E731
        launches_per_step = 3
        inputs = ((q, qh), (k, kh), (v, vh), (o, o.cpu().pin_memory()), (lse, lse.cpu().pin_memory()), (do, doh))
        outputs = grads[:3]
    elif w.direction == "fp8":
        signs_h = make_workload_signs(w).pin_memory()
        signs = signs_h.to(dev, non_blocking=True)
        ws8 = torch.empty(fa.fa_fwd_fp8_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
        step = lambda: fa.fa_fwd_fp8(q, k, v, signs, o, lse, scale=w.scale, causal=w.causal,  # noqa: E731
                                     workspace=ws8, stream=stream)
        launches_per_step = 2  # preparation (rotation + quantisation), attention
        inputs = ((q, qh), (k, kh), (v, vh))  # the rotation signs stay on the device
        outputs = (o, lse)
    else:
        step = lambda: fwd(q, k, v, o, lse, ws, stream)  # noqa: E731
        launches_per_step = 2 if w.n_splits > 1 else 1
        inputs = ((q, qh), (k, kh), (v, vh))
        outputs = (o, lse)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if fa.fa_status(clear=True) != 0:
        raise RuntimeError("device status word set during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(gpu_selector(dev))
    if rank == 0:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    launches = 0
    for i in range(args.steps):
        flush.zero_()  # write a buffer larger than L2 between timed launches
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        launches += launches_per_step
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.perf_counter()
    clocks = sampler.stop(t0, t1) if rank == 0 else None
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = reduce_max(sum(kernel_ms) / len(kernel_ms), world, dev)
    if fa.fa_status(clear=True) != 0:
        raise RuntimeError("device status word set during the timed region")

    # end to end through the public API: pinned host -> device, the step, device -> host.  The
    # one-split forward, the FP8 forward and the backward use fa_fwd_host / fa_fwd_fp8_host /
    # fa_bwd_host, which overlap the copies of one chunk of heads with the kernels of another
    # (the FP8 signs stay on the device); the other steps copy, run and copy back in turn.
    outputs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outputs]
    e2e_steps = max(1, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host_pipelined = w.direction == "fwd" and w.n_splits == 1
    for i in range(e2e_steps + 1):
        if i == 1:
            e0.record(stream)
        if host_pipelined:
            fa.fa_fwd_host(qh, kh, vh, outputs_h[0], outputs_h[1], q, k, v, o, lse, scale=w.scale,
                           causal=w.causal, stream=stream)
            continue
        if w.direction == "fp8":
            fa.fa_fwd_fp8_host(qh, kh, vh, outputs_h[0], outputs_h[1], q, k, v, signs, o, lse, ws8,
                               scale=w.scale, causal=w.causal, stream=stream)
            continue
        if w.direction == "bwd":
            fa.fa_bwd_host(tuple(h for _, h in inputs), tuple(outputs_h), tuple(dv for dv, _ in inputs),
                           tuple(outputs), grads[3], scale=w.scale, causal=w.causal, stream=stream)
            continue
        for dst, src in inputs:
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(outputs_h, outputs):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world, dev)
    if rank != 0:
        return

    flops = w.flops()
    metric, unit = metric_for(w)
    units = units_per_step(w)
    value = job_rate(units, ms, world)
    peak_tf, peak_gbs, peak_kind = peaks()
    if w.bound == "hbm":
        roofline = {"bound": "hbm", "achieved": units / (ms * 1e-3), "peak": peak_gbs, "unit": "GB/s",
                    "frac": units / (ms * 1e-3) / peak_gbs, "traffic": measured_traffic(w.name),
                    "peak_kind": f"HBM copy bandwidth, {peak_kind}",
                    "algorithmic_flops": flops, "algorithmic_bytes": w.algorithmic_bytes()}
    else:
        achieved = flops / (ms * 1e-3) / 1e12
        peak_label = f"bf16 dense burst, {peak_kind}"
        if w.direction == "fp8":  # E4M3 dense = the measured bf16 peak x 2 (nominal 4.5 / 2.25 PFLOP/s)
            peak_tf, peak_label = 2.0 * peak_tf, f"E4M3 dense = 2 x bf16 dense burst ({peak_kind})"
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": achieved / peak_tf, "traffic": measured_traffic(w.name),
                    "peak_kind": peak_label
                                 + {"bwd": "; timed over the step's three launches (D, dK/dV, dQ)",
                                    "fp8": "; timed over the step's two launches (rotation and quantisation, attention)"}
                                 .get(w.direction, ""),
                    "algorithmic_flops": flops, "algorithmic_bytes": w.algorithmic_bytes()}
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if w.direction == "fp8" else "bf16", "data": "synthetic",
        "config": workload_config(w),
        "roofline": roofline,
        "e2e": {"value": job_rate(units, e2e_ms, world), "unit": unit,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t, _ in inputs),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outputs)},
        "gpu_launches": launches,
        "clocks": clocks,
        "kernel_ms": {"min": min(kernel_ms), "median": statistics.median(kernel_ms), "max": max(kernel_ms)},
    }
    if world == 1 and not args.no_cpu_baseline:
        results = tuple(t.cpu() for t in (grads[:3] if w.direction == "bwd" else (o, lse)))
        line["cpu_baseline"], parity = cpu_baseline(w, results)
        if parity is not None:
            line["parity"] = parity
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
