"""The N > 1 bench path on CPU with gloo (world size 2): every rank runs its
own replica, the step time is the max over ranks, the value aggregates all
ranks' bytes, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [0.100 + 0.02 * rank, 0.150 - 0.01 * rank]
        got = bench.reduce_max(local, torch.device("cpu"))
        value = bench.whole_job_gbs(world, bench.algorithmic_bytes("bf16"), got[0])
        q.put((rank, got, value, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value, env in res:
        assert got == pytest.approx([0.12, 0.15])
        assert value == pytest.approx(2 * 542904324 / 0.12e-3 / 1e9)
        assert env == (2, rank, rank)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        fmt, steps, warmup, ref_rows = "bf16", 1, 3, 1

    assert bench.run_reference(A) is None
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes_of_the_headline():
    # K+V rows 128*2*2055*1024 + ids 128*2055*4 + q and out 2*128*24*512 + cu 129*4
    assert bench.algorithmic_bytes("bf16") == 542904324
    assert bench.algorithmic_bytes("fp8_e4m3") == 273551364 + 8  # + the two per-pool fp32 scales
    assert bench.algorithmic_bytes("int8") == 277760004
    assert bench.algorithmic_bytes("int4") == 143083524


def test_gpus_flag_launches_that_many_ranks():
    """--gpus 2 without a launcher re-runs the script under torch.distributed.run
    with two ranks (gloo on CPU here); the line reports n_gpus 2 and the slower
    rank's step time."""
    import json
    import subprocess
    import sys

    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    stub = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rank_stub.py")
    r = subprocess.run([sys.executable, stub, "--gpus", "2", "--steps", "3"], capture_output=True,
                       text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout            # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2
    assert line["ms_per_step"] >= 40.0          # rank 1's stand-in step: 40 ms
    assert line["ms_per_step"] > line["rank0_ms"] + 10.0
    assert line["value"] == pytest.approx(2 * 542904324 / (line["ms_per_step"] * 1e-3) / 1e9)
