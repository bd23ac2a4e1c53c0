"""bench.py's rank launcher and aggregation driven on CPU (used by
tests/test_multiproc.py; not a test file itself).

Run with --gpus N: without WORLD_SIZE in the environment it re-launches itself
under torch.distributed.run through bench.relaunch_ranks, exactly as bench.py
does; each rank joins the process group through bench.init_dist (gloo on CPU),
runs a stand-in step whose time grows with the rank, and the max over ranks
(bench.reduce_max) becomes the line's step time, which rank 0 prints with
n_gpus = the world size.
"""
import argparse
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    args = ap.parse_args()
    if bench.needs_relaunch(args.gpus):
        sys.exit(bench.relaunch_ranks(args.gpus, [os.path.abspath(__file__), *sys.argv[1:]]))
    ws, rank, local = bench.dist_env()
    dev = torch.device("cpu")
    bench.init_dist(dev)
    bench.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time.sleep(0.02 * (rank + 1))   # stand-in step: rank r takes (r + 1) * 20 ms
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    bench.barrier()
    step_ms = bench.reduce_max([ms], dev)[0]
    if rank == 0:
        print(json.dumps({"n_gpus": ws, "ms_per_step": step_ms, "rank0_ms": ms,
                          "value": bench.whole_job_gbs(ws, bench.algorithmic_bytes("bf16"), step_ms),
                          "scaling": "weak"}), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
