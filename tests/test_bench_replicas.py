"""The multi-rank host logic of bench.py on CPU: two gloo ranks (replicas
only, no data-path collective), max-over-ranks timing, whole-job throughput,
and the reference arm printing on rank 0 alone."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 1.0 + rank          # rank 1 is the slower one
    worst = bench.reduce_max(ms, world)
    value = bench.job_tflops(1e12, worst, world)
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"worst": worst, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()
    # reference arm: rank 0 prints one line, the other ranks return without work
    import contextlib
    import io
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "n128_d64"])
    with open(os.path.join(outdir, f"ref{rank}.txt"), "w") as f:
        f.write(buf.getvalue())


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["worst"] == r1["worst"] == 2.0
    assert r0["value"] == pytest.approx(2 * 1e12 / 2e-3 / 1e12)
    line = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    assert len(line) == 1
    rec = json.loads(line[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert (tmp_path / "ref1.txt").read_text() == ""
