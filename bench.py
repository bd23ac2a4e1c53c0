"""Benchmark: packed QSA decode at bs=128, L=2055, TP1 (24Q/2KV), D=256.

One step = one qsa_decode call over one batch (every selected K/V row
gathered, QK, softmax, PV, split merge). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--fmt bf16|fp8_e4m3|int8|int4|int8_g64|int4_g32|int8ring_int4]
                  [--impl native|reference] [--op decode|kv_write|topk]

The default bf16 line also carries `formats` (every quantised pool at the
headline shape), `small_batch` (batch sizes 1..64 of both topologies in the
short and saturated length bands, each call replayed from a CUDA graph) and
`topk` (the exact top-k + index expansion that produces the selected slots).

Timing: every timed region starts behind a few milliseconds of a clock-spin
kernel (torch.cuda._sleep), so all of its calls are queued before the GPU
reaches the start event and the events time the GPU, not the host's launch
rate. Clocks are read through NVML from a thread started before the warm-up.

--gpus N > 1 without a launcher re-runs this script under
torch.distributed.run with N ranks: independent replicas, one per GPU.

--impl reference times the FP64 CPU oracle on the host cores on a bounded
sample of the same workload (the deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import socket
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
SWEEP_SLOTS = 524288    # pool of the batch / length sweep
ROW_BYTES = {"bf16": 512, "fp8_e4m3": 256, "int8": 256, "int4": 128, "int8_g64": 256,
             "int4_g32": 128}
# per-row scale bytes: fp32 per (slot, KV head), or binary16 per channel group
SCALE_BYTES = {"bf16": 0, "fp8_e4m3": 0, "int8": 4, "int4": 4, "int8_g64": 8, "int4_g32": 16}
GATE_CYCLES = 20_000_000   # ~10 ms of clock spin at 2 GHz ahead of each timed region


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


def lengths_bytes(fmt: str, lengths, hq: int) -> int:
    """algorithmic_bytes for a batch of mixed lengths."""
    hkv = hq // 12
    n = int(sum(int(x) for x in lengths))
    bs = len(lengths)
    return (hkv * n * 2 * (ROW_BYTES[fmt] + SCALE_BYTES[fmt]) + n * 4 + 2 * bs * hq * 512
            + (bs + 1) * 4 + (8 if fmt == "fp8_e4m3" else 0))


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


def call_bytes(fmt: str, works, bs: int = BS) -> int:
    """Algorithmic bytes of one call of a saturated workload (tiered: the mean over
    the index sets, whose hot shares differ slightly)."""
    if fmt == I.TIERED:
        return sum(tiered_bytes(w) for w in works) // len(works)
    return algorithmic_bytes(fmt, bs=bs)


# ------------------------------------------------------------ ranks

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def needs_relaunch(gpus: int) -> bool:
    """True when N > 1 ranks were asked for but this process was not started by a
    launcher (no WORLD_SIZE in the environment)."""
    return gpus > 1 and "WORLD_SIZE" not in os.environ


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def relaunch_ranks(gpus: int, argv) -> int:
    """Run `argv` (a script and its arguments) under torch.distributed.run with one
    rank per GPU on this node; returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr=127.0.0.1", f"--master-port={free_port()}",
           *argv]
    return subprocess.call(cmd)


def init_dist(device):
    """Join the process group of a multi-rank run (NCCL with GPUs, gloo without)."""
    import torch.distributed as dist

    ws, _, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if device.type == "cuda" else "gloo")


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


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


# ------------------------------------------------------------ peaks, traffic

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


def measured_traffic(fmt: str, source: str = "qsa_decode.cu"):
    """DRAM bytes per launch from profiles/traffic.txt, if taken on the current kernel code."""
    src = os.path.join(ROOT, "sparse_attention_paged_qsa_gb300", "csrc", source)
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    key = kernel_source_key(src)
    for line in open(path):
        parts = line.split()
        if len(parts) == 3 and not line.startswith("#") and parts[0] == fmt and parts[2] == key:
            return int(parts[1])
    return None


# ------------------------------------------------------------ clocks

class Clocks:
    """SM clock and throttle reasons of one GPU, sampled from a thread, from before
    the warm-up until the last timed region ends. The first choice is NVML
    (libnvidia-ml, the library nvidia-smi reads), polled every millisecond: nothing
    is forked while kernels run. Without NVML, one long-running nvidia-smi process
    (-lms 100), started before the warm-up, is read instead. Each sample carries the
    host time it was taken at; summary(t0, t1) keeps those of one timed region."""

    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown")

    def __init__(self, device: torch.device, period_s: float = 0.001):
        self.device = device
        self.period = period_s
        self.samples = []            # (host time, sm MHz, max sm MHz, frozenset of reasons)
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.source = None

    # NVML ---------------------------------------------------------------
    def _nvml_open(self):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        vp, P = ctypes.c_void_p, ctypes.POINTER
        lib.nvmlDeviceGetHandleByUUID.argtypes = [ctypes.c_char_p, P(vp)]
        lib.nvmlDeviceGetHandleByPciBusId_v2.argtypes = [ctypes.c_char_p, P(vp)]
        lib.nvmlDeviceGetClockInfo.argtypes = [vp, ctypes.c_int, P(ctypes.c_uint)]
        lib.nvmlDeviceGetMaxClockInfo.argtypes = [vp, ctypes.c_int, P(ctypes.c_uint)]
        try:
            reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        reasons.argtypes = [vp, P(ctypes.c_ulonglong)]
        props = torch.cuda.get_device_properties(self.device)
        h = vp()
        ok = False
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(h)) == 0
        if not ok and hasattr(props, "pci_bus_id"):
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        if not ok:
            raise OSError("no NVML handle for this device")
        return lib, h, reasons

    def _nvml_loop(self, lib, h, reasons_fn):
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
                    and lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
                    and reasons_fn(h, ctypes.byref(rs)) == 0):
                active = frozenset(k for k, bit in self.REASONS.items() if rs.value & bit)
                self.samples.append((t, float(clk.value), float(mx.value), active))
            self._stop.wait(self.period)

    # nvidia-smi -----------------------------------------------------------
    def _smi_loop(self):
        for line in self._proc.stdout:
            t = time.perf_counter()
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) != 6:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            active = frozenset(k for k, v in zip(self.REASONS, parts[2:])
                               if "Active" in v and "Not" not in v)
            self.samples.append((t, sm, mx, active))

    def __enter__(self):
        try:
            lib, h, fn = self._nvml_open()
            self.source = "nvml"
            self._thread = threading.Thread(target=self._nvml_loop, args=(lib, h, fn), daemon=True)
        except (OSError, AttributeError):
            props = torch.cuda.get_device_properties(self.device)
            ident = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(
                self.device.index or 0)
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", ident, f"--query-gpu={self.SMI_FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                self._thread = threading.Thread(target=self._smi_loop, daemon=True)
            except OSError:
                self.source = None
        if self._thread is not None:
            self._thread.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=10)

    def summary(self, t0: float, t1: float):
        inside = [s for s in list(self.samples) if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source, "window_ms": (t1 - t0) * 1e3}
        sm = sorted(s[1] for s in inside)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(s[2] for s in inside),
                "sm_min_mhz": sm[0], "reasons": sorted(set().union(*(s[3] for s in inside))),
                "samples": len(inside), "source": self.source, "window_ms": (t1 - t0) * 1e3}


# ------------------------------------------------------------ timing

def gate():
    """Hold the current stream with torch's clock-spin kernel for a few milliseconds,
    so that the host queues every call of the timed region before the GPU reaches
    the region's start event."""
    torch.cuda._sleep(GATE_CYCLES)


def time_calls(launch, n: int, stream) -> float:
    """Milliseconds per call of n back-to-back calls launch(0..n-1) on `stream`, timed by
    CUDA events on that stream behind the gate; synchronised on both sides."""
    torch.cuda.synchronize()
    gate()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(n):
        launch(k)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def time_each(launch, n: int, stream):
    """Each call's own event pair (a diagnostic: the events between calls keep one
    call's launch from overlapping the previous call's tail)."""
    torch.cuda.synchronize()
    gate()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for k in range(n):
        evs[k][0].record(stream)
        launch(k)
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_graph(graph, n: int, stream) -> float:
    """Milliseconds per call of a captured graph of n calls, replayed once behind the gate."""
    torch.cuda.synchronize()
    gate()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def stats(xs):
    ys = sorted(xs)
    return {"min": ys[0], "median": ys[len(ys) // 2], "max": ys[-1]}


# ------------------------------------------------------------ reference arm

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


# ------------------------------------------------------------ the quantised pools

QUANT_FORMATS = ("fp8_e4m3", "int8", "int4", "int8_g64", "int4_g32", I.TIERED)


def measure_formats(args, dev, stream, scratch, peak):
    """Every quantised pool at the headline shape (bs=128, L=2055, 24Q/2KV): one pool
    per format, rotating index sets, back-to-back stream launches behind the gate."""
    import sparse_attention_paged_qsa_gb300 as qsa

    n = max(min(args.steps, 200), 1)
    res = {}
    for fmt in QUANT_FORMATS:
        works = make_workloads(fmt, 2, [100 + k for k in range(args.index_sets)], dev)
        w0 = works[0]
        out = torch.empty_like(w0.q)
        tier = {k: w0.extra[k] for k in I.TIER_KEYS} if fmt == I.TIERED else None
        meta = qsa.KVQuantMeta(fmt, L, w0.k_scale, w0.v_scale, w0.softmax_scale, 0, tier)

        def launch(k, works=works, meta=meta, out=out):
            w = works[k % len(works)]
            qsa.qsa_decode(w.q, w.k_pool, w.v_pool, meta, w.sel, w.cu, out, scratch, stream)

        for k in range(args.warmup):
            launch(k)
        ms = time_calls(launch, n, stream)
        b = call_bytes(fmt, works)
        res[fmt] = {"us_per_call": ms * 1e3, "calls_per_s": 1e3 / ms,
                    "gb_s": b / (ms * 1e-3) / 1e9, "pct_of_hbm_peak": 100.0 * b / (ms * 1e-3) / 1e9 / peak,
                    "bytes_per_call": b, "calls": n, "traffic": measured_traffic(fmt)}
        del works, w0, out, meta
        torch.cuda.empty_cache()
    if qsa.qsa_scratch_error(scratch):
        raise RuntimeError("device error flags after the quantised-pool runs")
    return res


# ------------------------------------------------------------ batch / length sweep

SWEEP_BATCHES = (1, 4, 16, 64)
SWEEP_BANDS = ("short", "medium", "saturated")


def measure_small_batches(args, dev, peak):
    """Batch sizes 1..64 of both topologies (TP1 24Q/2KV, TP2 12Q/1KV) over a bf16 pool
    of 524,288 slots, in the short (1-64), medium (512-1024) and saturated (2055)
    length bands. Each
    point's calls are captured in one CUDA graph (three index sets in turn) and
    replayed behind the gate, as a serving loop replays its decode."""
    import sparse_attention_paged_qsa_gb300 as qsa

    n = max(min(args.steps, 100), 1)
    out_rows = []
    for hkv in (2, 1):
        hq = 12 * hkv
        kc, vc, _, _ = I.make_pools(SWEEP_SLOTS, hkv, "bf16", seed=3, device=dev)
        for band in SWEEP_BANDS:
            lo, hi = I.BANDS[band]
            for bs in SWEEP_BATCHES:
                g = torch.Generator().manual_seed(1000 * bs + 10 * hkv + SWEEP_BANDS.index(band) + 1)
                sets = []
                for _ in range(args.index_sets):
                    lens = torch.randint(lo, hi + 1, (bs,), generator=g, dtype=torch.int64)
                    sel = I.uniform_indices(int(lens.sum()), SWEEP_SLOTS, g)
                    q = torch.randn(bs, hq, 256, generator=g).to(torch.bfloat16)
                    sets.append((q.to(dev), sel.to(dev), I.cu_from_lengths(lens).to(dev), lens))
                out = torch.empty(bs, hq, 256, dtype=torch.bfloat16, device=dev)
                scratch = qsa.alloc_scratch(bs, hq, hi, dev)
                meta = qsa.KVQuantMeta("bf16", hi, None, None, I.SOFTMAX_SCALE)
                gs = torch.cuda.Stream(device=dev)
                gs.wait_stream(torch.cuda.current_stream())

                def launch(k, st):
                    q, sel, cu, _ = sets[k % len(sets)]
                    qsa.qsa_decode(q, kc, vc, meta, sel, cu, out, scratch, st)

                with torch.cuda.stream(gs):
                    for k in range(args.warmup):
                        launch(k, gs)
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=gs):
                    for k in range(n):
                        launch(k, gs)
                with torch.cuda.stream(gs):
                    ms = time_graph(graph, n, gs)
                if qsa.qsa_scratch_error(scratch):
                    raise RuntimeError(f"device error flags at bs={bs} hkv={hkv} {band}")
                nbytes = sum(lengths_bytes("bf16", sets[k % len(sets)][3].tolist(), hq)
                             for k in range(n)) / n
                toks = sum(int(sets[k % len(sets)][3].sum()) for k in range(n)) / n
                rows_b = sum(int(s[3].sum()) for s in sets) * hkv * 1024
                out_rows.append({
                    "topology": "TP1 24Q/2KV" if hkv == 2 else "TP2 12Q/1KV", "bs": bs,
                    "band": f"{band} {lo}-{hi}", "us_per_call": ms * 1e3,
                    "calls_per_s": 1e3 / ms, "tokens_per_s": toks / (ms * 1e-3),
                    "gb_s": nbytes / (ms * 1e-3) / 1e9,
                    "pct_of_hbm_peak": 100.0 * nbytes / (ms * 1e-3) / 1e9 / peak,
                    "l2": "L2-warm" if rows_b <= 129e6 else "larger than L2"})
                del graph, scratch, out, sets
        del kc, vc
        torch.cuda.empty_cache()
    return out_rows


# ------------------------------------------------------------ top-k + index expansion

TOPK_PAGE = 64


def topk_bytes(bs: int, cap: int, ratio: int, topk: int) -> int:
    """Bytes one qsa_topk_expand call must move with full contexts of `cap` tokens:
    every block score once, the context lengths, one page-table entry per kept block
    or tail page, the packed slot ids written and cu_seqlens."""
    nb = cap // ratio
    kb = min(nb, topk // ratio)
    row = ratio * kb + cap % ratio
    pages = kb + (1 if cap % ratio else 0)
    return bs * (nb * 4 + 4 + pages * 4 + row * 4) + (bs + 1) * 4


def measure_topk(args, dev, peak):
    """qsa_topk_expand at the pages' sizes (token_topk 2048 -- 2032 at ratio 16, whose rows
    must fit the decode's 2055 --, compress ratios 4 / 8 / 16,
    8K and 256K-token contexts, bs 1 and 128, through a 64-token page table): two
    sets of N(0,1) block scores in turn, back-to-back stream launches behind the gate."""
    import sparse_attention_paged_qsa_gb300 as qsa

    n = max(min(args.steps, 200), 1)
    stream = torch.cuda.current_stream()
    rows = []
    only = getattr(args, "topk_point", None)
    for cap in (8192, I.TOPK_CAPACITY):
        for bs in (1, BS):
            for ratio in (4, 8, 16):
                if only is not None and (cap, bs, ratio) != only:
                    continue
                topk = I.topk_budget(ratio)
                sets = [I.block_scores(bs, cap // ratio, 100 + k, dev, specials=False)
                        for k in range(2)]
                lens = torch.full((bs,), cap, dtype=torch.int32, device=dev)
                pt = I.page_table(bs, cap, TOPK_PAGE, 7, dev)
                sel = torch.empty(bs * (topk + ratio - 1), dtype=torch.int32, device=dev)
                cu = torch.empty(bs + 1, dtype=torch.int32, device=dev)

                def launch(k, sets=sets, lens=lens, pt=pt, sel=sel, cu=cu, ratio=ratio, cap=cap):
                    qsa.qsa_topk_expand(sets[k % 2], lens, sel, cu, topk, ratio, cap,
                                        page_table=pt, page_size=TOPK_PAGE, stream=stream)

                for k in range(args.warmup):
                    launch(k)
                ms = time_calls(launch, n, stream)
                b = topk_bytes(bs, cap, ratio, topk)
                rows.append({"context": cap, "bs": bs, "compress_ratio": ratio, "token_topk": topk,
                             "us_per_call": ms * 1e3, "calls_per_s": 1e3 / ms,
                             "gb_s": b / (ms * 1e-3) / 1e9,
                             "pct_of_hbm_peak": 100.0 * b / (ms * 1e-3) / 1e9 / peak,
                             "bytes_per_call": b})
                del sets, lens, pt, sel, cu
    torch.cuda.empty_cache()
    return rows


def run_topk(args):
    """The top-k + index expansion alone: one JSON line (bs=128, 256K contexts, ratio 4
    as the value; every measured point under `points`)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = measured_peaks()
    clk = Clocks(dev).__enter__()
    t0 = time.perf_counter()
    pts = measure_topk(args, dev, peak)
    clocks = clk.summary(t0, time.perf_counter())
    clk.__exit__()
    if not pts:
        raise SystemExit("--topk-point names no measured point (capacities 8192 / 262144, "
                         "bs 1 / 128, ratios 4 / 8 / 16)")
    head = next((p for p in pts if p["context"] == I.TOPK_CAPACITY and p["bs"] == BS
                 and p["compress_ratio"] == 4), pts[0])
    print(json.dumps({
        "metric": "qsa_topk_expand calls/s (exact top-k 2048 tokens + index expansion, 256K contexts)",
        "op": "topk", "value": head["calls_per_s"], "unit": "calls/s", "n_gpus": 1,
        "steps": max(min(args.steps, 200), 1), "warmup": args.warmup,
        "ms_per_step": head["us_per_call"] * 1e-3, "higher_is_better": True, "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": f"bs={head['bs']}, {head['context']}-token contexts, compress ratio "
                               f"{head['compress_ratio']}, token_topk {head['token_topk']}, "
                               "64-token page table"},
        "roofline": {"bound": "hbm", "achieved": head["gb_s"], "peak": peak, "unit": "GB/s",
                     "frac": head["gb_s"] / peak, "peak_source": f"{kind} hbm_gbs",
                     "bytes_per_launch": head["bytes_per_call"],
                     "traffic": measured_traffic(
                         f"topk_{head['context']}_bs{head['bs']}_r{head['compress_ratio']}", "qsa_topk.cu")},
        "points": pts, "clocks": clocks}), flush=True)


# ------------------------------------------------------------ the headline

def run_native(args):
    import sparse_attention_paged_qsa_gb300 as qsa

    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)  # before the process group, so NCCL binds this rank's GPU
    init_dist(dev)
    fmt = args.fmt
    bs = args.bs
    clk = Clocks(dev).__enter__()
    works = make_workloads(fmt, 2 + rank, [100 + 7 * rank + k for k in range(args.index_sets)], dev,
                           bs=bs)
    w0 = works[0]
    out = torch.empty_like(w0.q)
    scratch = qsa.alloc_scratch(bs, HQ, L, dev)
    tier = {k: w0.extra[k] for k in I.TIER_KEYS} if fmt == I.TIERED else None
    meta = qsa.KVQuantMeta(fmt, L, w0.k_scale, w0.v_scale, w0.softmax_scale, 0, tier)
    stream = torch.cuda.current_stream()
    grid = qsa.qsa_decode_grid(bs, HQ, L)

    def step(k, st=stream):
        w = works[k % len(works)]
        qsa.qsa_decode(w.q, w.k_pool, w.v_pool, meta, w.sel, w.cu, out, scratch, st)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    barrier()
    graph = None
    if args.graph:  # the timed calls as one CUDA graph
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for k in range(args.steps):
                step(k, gs)
        torch.cuda.synchronize()
        barrier()
    t_win0 = time.perf_counter()
    if graph is not None:
        step_ms = time_graph(graph, args.steps, stream)
    else:  # one stream launch per call; each may begin as its predecessor drains
        step_ms = time_calls(step, args.steps, stream)
    t_win1 = time.perf_counter()
    barrier()
    clocks = clk.summary(t_win0, t_win1)
    if qsa.qsa_scratch_error(scratch):
        raise RuntimeError("device error flags after the timed calls")
    # diagnostic: the same calls each between its own pair of events
    per_call = None if args.no_per_call else time_each(step, min(args.steps, 200), stream)

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
        gate()
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

    step_ms, e2e_ms = reduce_max([step_ms, e2e_ms if e2e_steps else 0.0], dev)
    abytes = call_bytes(fmt, works, bs)
    value = whole_job_gbs(ws, abytes, step_ms)
    e2e_val = whole_job_gbs(ws, abytes, e2e_ms) if e2e_steps else None
    achieved = abytes / (step_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    calls = ws / (step_ms * 1e-3)
    rows_bytes = bs * HKV * L * 2 * (ROW_BYTES.get(fmt, 0) + SCALE_BYTES.get(fmt, 0))

    extras = not args.no_extras and ws == 1 and fmt == "bf16" and bs == BS
    formats = small = topk = None
    if extras:
        formats = measure_formats(args, dev, stream, scratch, peak)
        small = measure_small_batches(args, dev, peak)
        topk = measure_topk(args, dev, peak)

    cpu = None
    if rank == 0 and args.cpu_rows > 0:
        import oracle

        oracle.build()
        cpu = cpu_baseline(fmt, min(args.cpu_rows, bs), works[0], call_bytes=abytes, bs=bs)
    clk.__exit__()

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
                                  else "one stream launch per call, all queued behind a "
                                       "clock-spin gate before the start event")},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "bytes_per_launch": abytes, "kernel_ms": step_ms},
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms} if e2e_steps else None,
            "gpu_launches": args.steps,
            "clocks": clocks,
            "per_call_ms": stats(per_call) if per_call else None,
            "cpu_baseline": cpu,
        }
        if formats is not None:
            line["formats"] = formats
        if small is not None:
            line["small_batch"] = small
        if topk is not None:
            line["topk"] = topk
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------ the KV write

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
    clk = Clocks(dev).__enter__()
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
    t0 = time.perf_counter()
    ms = time_calls(step, args.steps, stream)
    clocks = clk.summary(t0, time.perf_counter())
    clk.__exit__()
    if int(err.item()):
        raise RuntimeError("device error flag set")
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
        "gpu_launches": args.steps * (2 if tier is not None else 1), "clocks": clocks}),
        flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)  # ~0.27 s timed
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--fmt", default="bf16", choices=list(I.FORMATS) + [I.TIERED])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--op", default="decode", choices=["decode", "kv_write", "topk"],
                    help="decode (the headline), the quantising KV write, or the top-k + "
                         "index expansion")
    ap.add_argument("--index-sets", type=int, default=3)
    ap.add_argument("--bs", type=int, default=BS,
                    help="sequences per call (the headline is 128; smaller for latency)")
    ap.add_argument("--graph", action="store_true",
                    help="time the calls captured in one CUDA graph")
    ap.add_argument("--no-per-call", action="store_true",
                    help="skip the diagnostic that times each call between its own pair of events")
    ap.add_argument("--cpu-rows", type=int, default=128,
                    help="sequences of the oracle CPU-baseline sample (0 disables)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the quantised-pool and small-batch objects of the default line")
    ap.add_argument("--ref-rows", type=int, default=8,
                    help="sequences per step of the --impl reference sample")
    ap.add_argument("--topk-point", default=None, metavar="CAPACITY,BS,RATIO",
                    help="--op topk: measure this point only (e.g. 262144,128,4)")
    args = ap.parse_args(argv)
    if args.topk_point is not None:
        try:
            cap, bs, ratio = (int(x) for x in args.topk_point.split(","))
        except ValueError:
            ap.error("--topk-point takes CAPACITY,BS,RATIO")
        args.topk_point = (cap, bs, ratio)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def main():
    args = parse_args()
    if needs_relaunch(args.gpus):
        sys.exit(relaunch_ranks(args.gpus, [os.path.abspath(__file__), *sys.argv[1:]]))
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "kv_write":
        run_kv_write(args)
    elif args.op == "topk":
        run_topk(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
