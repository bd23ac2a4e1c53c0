"""Host logic of the measurement (no GPU): the algorithmic bytes every bench line
divides by, the DRAM-traffic lookup keyed to the kernel source, and the JSON
contract of the reference arm."""
import json
import os

import pytest
import torch

import bench
from sparse_attention_paged_qsa_gb300 import inputs as I


def test_algorithmic_bytes_of_the_grouped_pools():
    rows = 128 * 2 * 2055 * 2  # selected (id, KV head) rows, K and V
    rest = 128 * 2055 * 4 + 2 * 128 * 24 * 512 + 129 * 4  # ids, q and out, cu_seqlens
    # int8 codes + four binary16 scales per row; int4 nibbles + eight binary16 scales
    assert bench.algorithmic_bytes("int8_g64") == rows * (256 + 4 * 2) + rest
    assert bench.algorithmic_bytes("int4_g32") == rows * (128 + 8 * 2) + rest
    # sizes scale with the batch, the length and the head count as the formula says
    assert bench.algorithmic_bytes("bf16", bs=1, length=1, hq=12) == 1 * 1 * 1 * 2 * 512 + 4 + 2 * 12 * 512 + 2 * 4


def test_tiered_bytes_count_the_hot_rows():
    w = I.tiered(seed=40, bs=3, num_slots=4096, ring_slots=256, lengths=[7, 300, 64], hot_share=0.5)
    owner = w.extra["owner"].long()
    hot = sum(int(owner[s & 255]) == s for s in w.sel.long().tolist())  # brute force over ids
    n = w.sel.numel()
    per_head = hot * 2 * (256 + 8) + (n - hot) * 2 * (128 + 16) + n * 4
    expect = 2 * per_head + n * 4 + 2 * 3 * 24 * 512 + 4 * 4
    assert 0 < hot < n
    assert bench.tiered_bytes(w) == expect


def test_traffic_lookup_is_keyed_to_the_kernel_source(tmp_path, monkeypatch):
    src_dir = tmp_path / "sparse_attention_paged_qsa_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "qsa_decode.cu"
    src.write_text("int f() { return 1; } // v1\n")
    key = bench.kernel_source_key(str(src))
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"# comment\nbf16 123 {key}\nint8 456 {'0' * 64}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("bf16") == 123
    assert bench.measured_traffic("int8") is None      # taken on other code
    assert bench.measured_traffic("fp8_e4m3") is None  # never taken
    src.write_text("/* a new comment */\nint f()  {\n  return 1;\n}  // v2\n")
    assert bench.measured_traffic("bf16") == 123       # comments and layout only
    src.write_text("int f() { return 2; } // v1\n")   # the code changed since
    assert bench.measured_traffic("bf16") is None


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)

    class A:
        fmt, steps, warmup, ref_rows = "int8", 1, 3, 1

    bench.run_reference(A)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["value"] > 0 and line["config"]["workload"].startswith("packed QSA decode bs=128")
