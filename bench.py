"""Benchmark: packed QSA decode at bs=128, L=2055, TP1 (24Q/2KV), D=256.

One step = one qsa_decode call over one batch (every selected K/V row
gathered, QK, softmax, PV, split merge). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--fmt bf16|fp8_e4m3|int8|int4|int8_g64|int4_g32|int8ring_int4]
                  [--impl native|reference]

--impl reference times the FP64 CPU oracle on the host cores on a bounded
sample of the same workload (the deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_paged_qsa_gb300 import inputs as I  # noqa: E402

METRIC = "selected-KV HBM GB/s (% of GB300 peak) & qsa_decode calls/s at bs=128, L=2055"
BS, L, HQ, HKV, SLOTS = 128, I.MAX_CAPACITY, 24, 2, 1048576
ROW_BYTES = {"bf16": 512, "fp8_e4m3": 256, "int8": 256, "int4": 128, "int8_g64": 256,
             "int4_g32": 128}
# per-row scale bytes: fp32 per (slot, KV head), or binary16 per channel group
SCALE_BYTES = {"bf16": 0, "fp8_e4m3": 0, "int8": 4, "int4": 4, "int8_g64": 8, "int4_g32": 16}


def algorithmic_bytes(fmt: str, bs: int = BS, length: int = L, hq: int = HQ) -> int:
    """Bytes one call must move: every selected K and V row (with its per-slot
    scales), the slot ids, q, out and cu_seqlens (per-pool fp8 scales: 8 B)."""
    hkv = hq // 12
    kv = bs * hkv * length * 2 * (ROW_BYTES[fmt] + SCALE_BYTES[fmt])
    idx = bs * length * 4
    q = out = bs * hq * 256 * 2
    cu = (bs + 1) * 4
    extra = 8 if fmt == "fp8_e4m3" else 0
    return kv + idx + q + out + cu + extra


TIER_HOT_SHARE = 0.25   # share of each selection drawn from slots that own their ring row


def tiered_bytes(work) -> int:
    """Bytes one tiered call must move: per selected (id, KV head) the owner entry
    (4 B) and, for K and V, the ring row with its 4 binary16 scales (264 B) when the
    slot owns its ring position, else the int4_g32 row with its 8 scales (144 B);
    plus slot ids, q, out and cu_seqlens."""
    sel = work.sel.long()
    owner = work.extra["owner"].long()
    hot = int((owner[sel & (owner.numel() - 1)] == sel).sum())
    n = sel.numel()
    hkv = work.num_kv_heads
    kv = hkv * (hot * 2 * 264 + (n - hot) * 2 * 144 + n * 4)
    return kv + n * 4 + 2 * work.bs * work.num_q_heads * 512 + (work.bs + 1) * 4


def oracle_decode(w, threads: int = 0):
    import oracle

    if w.fmt == I.TIERED:
        t = w.extra
        return oracle.decode_tiered(w.q, w.k_pool, w.v_pool, w.sel, w.cu, w.softmax_scale,
                                    w.k_scale, w.v_scale, t["k_ring"], t["v_ring"],
                                    t["k_ring_scale"], t["v_ring_scale"], t["owner"],
                                    threads=threads)
    return oracle.decode(w.q, w.k_pool, w.v_pool, w.fmt, w.sel, w.cu, w.softmax_scale,
                         w.k_scale, w.v_scale, threads=threads)


def make_workloads(fmt: str, seed: int, index_seeds, device, bs: int = BS, num_slots: int = SLOTS):
    """The saturated config's workloads (one pool, several index sets) for a format."""
    if fmt == I.TIERED:
        ring = min(I.RING_SLOTS, num_slots)
        pools = I.make_tiered_pools(num_slots, HKV, ring, seed, device=device)
        return [I.tiered(seed=s, device=device, bs=bs, num_slots=num_slots, ring_slots=ring,
                         lengths=[L] * bs, hot_share=TIER_HOT_SHARE, pools=pools)
                for s in index_seeds]
    pools = I.make_pools(num_slots, HKV, fmt, seed=seed, device=device)
    return [I.tp1_saturated(seed=seed, device=device, fmt=fmt, bs=bs, index_seed=s, pools=pools)
            for s in index_seeds]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(values, device):
    """Element-wise max of a list of floats over all ranks (identity when not distributed)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_gbs(world: int, bytes_per_rank_step: int, step_ms: float) -> float:
    """Aggregate GB/s: every rank moves its own bytes per step; time is the slowest rank's."""
    return world * bytes_per_rank_step / (step_ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_key(path: str) -> str:
    """sha256 of a CUDA source with its comments and whitespace removed: a key that
    changes when the code does, not when a comment does (no string literal in the
    kernel sources contains a comment marker)."""
    import hashlib
    import re

    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


def measured_traffic(fmt: str):
    """DRAM bytes per launch from profiles/traffic.txt, if taken on the current kernel code."""
    src = os.path.join(ROOT, "sparse_attention_paged_qsa_gb300", "csrc", "qsa_decode.cu")
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    key = kernel_source_key(src)
    for line in open(path):
        parts = line.split()
        if len(parts) == 3 and not line.startswith("#") and parts[0] == fmt and parts[2] == key:
            return int(parts[1])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
                parts = [p.strip() for p in out.stdout.strip().split(",")]
                if len(parts) == 6:
                    self.samples.append(parts)
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = sorted(float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit())
        mx = max((float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if "Active" in s[2 + i] and "Not" not in s[2 + i]})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(self.samples)}


def cpu_baseline(fmt: str, sample_rows: int, work, threads: int = 0, call_bytes: int = 0,
                 bs: int = BS):
    """Time the FP64 oracle on `sample_rows` sequences of the workload; returns a dict."""
    import oracle

    sub = I.host_subset(work, list(range(sample_rows)))
    t0 = time.perf_counter()
    oracle_decode(sub, threads=threads)
    dt = time.perf_counter() - t0
    b = (call_bytes or algorithmic_bytes(fmt, bs=bs)) * sample_rows // bs
    return {"value": b / dt / 1e9, "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle", "calls_per_s": (sample_rows / bs) / dt,
            "sample": f"{sample_rows} of {bs} sequences (L={L}, 24Q/2KV), {dt:.2f} s, "
                      "scaled to bytes of the full call"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    gen_dev = "cpu"
    rows = args.ref_rows
    # host-only generation of exactly the sampled sequences' data
    w = make_workloads(args.fmt, 2, [2], gen_dev, bs=rows, num_slots=SLOTS // 8)[0]
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle_decode(w)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    dt = sum(times) / len(times)
    b = tiered_bytes(w) if args.fmt == I.TIERED else algorithmic_bytes(args.fmt, bs=rows)
    gbs = b / dt / 1e9
    calls = (rows / BS) / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "calls_per_s": calls, "tokens_per_s": calls * BS * L,
        "config": {"workload": f"packed QSA decode bs={BS} L={L} 24Q/2KV D=256 {args.fmt} pool",
                   "sample_sequences_per_step": rows, "pool_slots": SLOTS // 8},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{rows} of {BS} sequences per step, scaled by bytes"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_native(args):
    import sparse_attention_paged_qsa_gb300 as qsa

    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)  # before the process group, so NCCL binds this rank's GPU
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    fmt = args.fmt
    bs = args.bs
    works = make_workloads(fmt, 2 + rank, [100 + 7 * rank + k for k in range(args.index_sets)], dev,
                           bs=bs)
    w0 = works[0]
    out = torch.empty_like(w0.q)
    scratch = qsa.alloc_scratch(bs, HQ, L, dev)
    tier = {k: w0.extra[k] for k in I.TIER_KEYS} if fmt == I.TIERED else None
    meta = qsa.KVQuantMeta(fmt, L, w0.k_scale, w0.v_scale, w0.softmax_scale, 0, tier)
    stream = torch.cuda.current_stream()
    grid = qsa.qsa_decode_grid(bs, HQ, L)

    def step(k):
        w = works[k % len(works)]
        qsa.qsa_decode(w.q, w.k_pool, w.v_pool, meta, w.sel, w.cu, out, scratch, stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    graph = None
    if args.graph:  # the timed calls as one CUDA graph: no host time between launches
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for k in range(args.steps):
                qsa.qsa_decode(works[k % len(works)].q, w0.k_pool, w0.v_pool, meta,
                               works[k % len(works)].sel, works[k % len(works)].cu, out, scratch, gs)
        torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        ev[0].record(stream)
        if graph is not None:
            graph.replay()
        else:  # no stream work between the calls: each launch may begin as its predecessor drains
            for k in range(args.steps):
                step(k)
        ev[-1].record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = ev[0].elapsed_time(ev[-1])
    per = [total_ms / args.steps]
    err = qsa.qsa_scratch_error(scratch)
    if err:
        raise RuntimeError(f"device error flags {err}")

    # e2e: host (pinned) q / slot ids / cu_seqlens -> device, decode, output -> host,
    # every step. Device inputs and outputs are double-buffered over three streams
    # (copy in, compute, copy out), as a serving loop would run them: step k+1's
    # inputs land while step k computes, and step k's output returns meanwhile.
    e2e_steps = args.steps if not args.no_e2e else 0
    hq_ = [w.q.cpu().pin_memory() for w in works]
    hsel = [w.sel.cpu().pin_memory() for w in works]
    hcu = [w.cu.cpu().pin_memory() for w in works]
    hout = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    dq = [torch.empty_like(w0.q) for _ in range(2)]
    dsel = [torch.empty_like(w0.sel) for _ in range(2)]
    dcu = [torch.empty_like(w0.cu) for _ in range(2)]
    dout = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]   # inputs of buffer j copied in
    computed = [torch.cuda.Event() for _ in range(2)]   # decode of buffer j done
    drained = [torch.cuda.Event() for _ in range(2)]    # output of buffer j copied out
    for j in range(2):
        drained[j].record(stream)

    def e2e_step(k):
        j, b = k % len(works), k % 2
        s_in.wait_event(drained[b])        # the buffer's previous decode and copy-out are done
        with torch.cuda.stream(s_in):
            dq[b].copy_(hq_[j], non_blocking=True)
            dsel[b].copy_(hsel[j], non_blocking=True)
            dcu[b].copy_(hcu[j], non_blocking=True)
        in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        qsa.qsa_decode(dq[b], w0.k_pool, w0.v_pool, meta, dsel[b], dcu[b], dout[b], scratch, stream)
        computed[b].record(stream)
        s_out.wait_event(computed[b])
        with torch.cuda.stream(s_out):
            hout[b].copy_(dout[b], non_blocking=True)
        drained[b].record(s_out)

    e2e_ms = float("nan")
    if e2e_steps:
        for k in range(args.warmup):
            e2e_step(k)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)  # nothing of the timed steps starts before e0
        for k in range(e2e_steps):
            e2e_step(k)
        stream.wait_stream(s_out)  # ... and e1 follows the last copy out
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = hq_[0].numel() * 2 + hsel[0].numel() * 4 + hcu[0].numel() * 4
    d2h = hout[0].numel() * 2

    step_ms = total_ms / args.steps
    step_ms, e2e_ms = reduce_max([step_ms, e2e_ms if e2e_steps else 0.0], dev)
    if fmt == I.TIERED:  # the bytes depend on which rows are hot: the mean over the index sets
        abytes = sum(tiered_bytes(w) for w in works) // len(works)
    else:
        abytes = algorithmic_bytes(fmt, bs=bs)
    value = whole_job_gbs(ws, abytes, step_ms)
    e2e_val = whole_job_gbs(ws, abytes, e2e_ms) if e2e_steps else None
    kernel_ms = sum(per) / len(per)
    achieved = abytes / (kernel_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    calls = ws / (step_ms * 1e-3)
    rows_bytes = bs * HKV * L * 2 * (ROW_BYTES.get(fmt, 0) + SCALE_BYTES.get(fmt, 0))

    cpu = None
    if rank == 0 and args.cpu_rows > 0:
        import oracle

        oracle.build()
        cpu = cpu_baseline(fmt, min(args.cpu_rows, bs), works[0], call_bytes=abytes, bs=bs)

    if rank == 0:
        traffic = measured_traffic(fmt)
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": fmt, "data": "synthetic",
            "calls_per_s": calls, "tokens_per_s": calls * bs * L,
            "pct_of_hbm_peak": 100.0 * achieved / peak,
            "config": {"workload": f"packed QSA decode bs={bs} L={L} 24Q/2KV D=256 {fmt} pool"
                                   + (f" (ring {I.RING_SLOTS}, {TIER_HOT_SHARE:.0%} of ids hot)"
                                      if fmt == I.TIERED else ""),
                       "pool_slots": SLOTS, "index_sets": args.index_sets, "grid_ctas": grid,
                       "l2": ("inputs larger than L2: 538 MB of K/V rows per call from a 2 GiB "
                              "pool, rotating index sets" if bs == BS else
                              f"{rows_bytes / 1e6:.0f} MB of K/V rows per index set x "
                              f"{args.index_sets} sets: " + ("larger than L2" if rows_bytes *
                              args.index_sets > 129e6 else "L2-warm (fits in the 129 MB L2)")),
                       "parallelism": f"replicas x{ws}",
                       "launch": ("the timed calls replayed as one CUDA graph" if args.graph
                                  else "one stream launch per call")},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "bytes_per_launch": abytes, "kernel_ms": kernel_ms},
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms} if e2e_steps else None,
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


KVW_TOKENS = 131072  # one prefill chunk: 128 sequences x 1024 new tokens


def kv_write_bytes(fmt: str, n: int = KVW_TOKENS, hkv: int = HKV, ring_rows: int = 0) -> int:
    """Bytes one qsa_kv_write call must move: the new bf16 K and V rows, the slot
    ids, the written codes and (int8/int4) the written per-row scales. Tiered: the
    int4_g32 rows of every token, plus for each ring position the write claims
    (`ring_rows` of them) its int8_g64 rows with scales and its owner entry."""
    read = 2 * n * hkv * 512 + n * 4 + (8 if fmt == "fp8_e4m3" else 0)
    if fmt == I.TIERED:
        return read + 2 * n * hkv * (128 + 16) + ring_rows * (2 * hkv * (256 + 8) + 4)
    write = 2 * n * hkv * (ROW_BYTES[fmt] + SCALE_BYTES[fmt])
    return read + write


def run_kv_write(args):
    """Secondary measurement: the quantising KV write (one call per step)."""
    import sparse_attention_paged_qsa_gb300 as qsa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fmt = args.fmt
    tier = None
    if fmt == I.TIERED:
        kc, vc, ks, vs, tier = I.make_tiered_pools(SLOTS, HKV, I.RING_SLOTS, 2, device=dev)
    else:
        kc, vc, ks, vs = I.make_pools(SLOTS, HKV, fmt, seed=2, device=dev)
    g = torch.Generator(device=dev).manual_seed(7)
    xs = [torch.randn(KVW_TOKENS, HKV, 256, generator=g, device=dev).to(torch.bfloat16)
          for _ in range(4)]
    slots = [torch.randperm(SLOTS, generator=g, device=dev)[:KVW_TOKENS].to(torch.int32)
             for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(k):
        if tier is not None:
            qsa.qsa_kv_write_tiered(xs[k % 4], xs[(k + 1) % 4], slots[k % 2], kc, vc, ks, vs, tier,
                                    err, stream)
        else:
            qsa.qsa_kv_write(fmt, xs[k % 4], xs[(k + 1) % 4], slots[k % 2], kc, vc, ks, vs, err,
                             stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        e0.record(stream)
        for k in range(args.steps):
            step(k)
        e1.record(stream)
        torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError("device error flag set")
    ms = e0.elapsed_time(e1) / args.steps
    ring_rows = 0
    if tier is not None:  # ring positions each write claims (the same two slot sets alternate)
        ring_rows = sum(int(torch.unique(sl.long() & (I.RING_SLOTS - 1)).numel()) for sl in slots) // 2
    b = kv_write_bytes(fmt, ring_rows=ring_rows)
    gbs = b / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    print(json.dumps({
        "metric": "quantising KV write HBM GB/s (128 x 1024 new tokens, 24Q/2KV, D=256)",
        "op": "kv_write", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": fmt,
        "data": "synthetic", "tokens_per_s": KVW_TOKENS / (ms * 1e-3),
        "config": {"workload": f"kv write of {KVW_TOKENS} tokens x 2 KV heads into a "
                               f"{SLOTS}-slot {fmt} pool, random distinct slots"
                               + (f", {I.RING_SLOTS}-row ring" if tier is not None else "")},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": f"{kind} hbm_gbs", "bytes_per_launch": b},
        "gpu_launches": args.steps, "clocks": clk.summary()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)  # ~0.3 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--fmt", default="bf16", choices=list(I.FORMATS) + [I.TIERED])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--op", default="decode", choices=["decode", "kv_write"],
                    help="decode (the headline) or the quantising KV write")
    ap.add_argument("--index-sets", type=int, default=3)
    ap.add_argument("--bs", type=int, default=BS,
                    help="sequences per call (the headline is 128; smaller for latency)")
    ap.add_argument("--graph", action="store_true",
                    help="time the calls captured in one CUDA graph (no host gaps between them)")
    ap.add_argument("--cpu-rows", type=int, default=128,
                    help="sequences of the oracle CPU-baseline sample (0 disables)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--ref-rows", type=int, default=8,
                    help="sequences per step of the --impl reference sample")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "kv_write":
        run_kv_write(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
