"""CUDA-graph replay sweep: lengths and slot ids change on the device between
replays, the captured decode reads them there (sglang PR #36845, "Changes":
captured graphs replay with changed cu_seqlens without host readback).

Each (topology, batch size, length band) graph is captured once and replayed
1000 times. Every replay regenerates cu_seqlens and the packed slot ids with a
counter-based hash of (seed, replay, b, j) inside the graph, runs qsa_decode,
and checks on the device that the split counters are back to zero and that
live rows are finite and non-zero. Sampled replays are also compared with the
oracle on sampled sequences (inputs regenerated on the host by the same
function). A second stress test runs 150,000 launches and checks the counters.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import REL_L2_TOL, counters, rel_l2

pytestmark = pytest.mark.gpu

SEED = 3
SLOTS = 524288
BATCHES = list(range(1, 17)) + [24, 32, 48, 64, 96, 128]
REPLAYS = 1000
CHECK_EVERY = 100


def _sweep_topology(dev, hq):
    hkv = hq // 12
    kc, vc, _, _ = I.make_pools(SLOTS, hkv, "bf16", SEED, device=dev)
    k_host, v_host = kc.cpu(), vc.cpu()
    worst = 0.0
    for band in ("short", "medium", "saturated"):
        cap = I.BANDS[band][1]
        for bs in BATCHES:
            q = I.make_query(bs, hq, SEED * 7 + bs, device=dev)
            sel = torch.zeros(bs * cap, dtype=torch.int32, device=dev)
            cu = torch.zeros(bs + 1, dtype=torch.int32, device=dev)
            out = torch.zeros(bs, hq, 256, dtype=torch.bfloat16, device=dev)
            scratch = qsa.alloc_scratch(bs, hq, cap, dev)
            ly = qsa.qsa_decode_scratch_layout(bs, hq, cap)
            cnt = scratch[ly["counters_offset"]:ly["counters_offset"] + 4 * ly["counters_count"]].view(
                torch.int32)
            meta = qsa.KVQuantMeta("bf16", cap, None, None, 1 / 16)
            replay = torch.zeros(1, dtype=torch.int64, device=dev)
            bad = torch.zeros(1, dtype=torch.int32, device=dev)

            def body():
                I.replay_inputs(SEED, replay, bs, band, cap, SLOTS, sel, cu)
                qsa.qsa_decode(q, kc, vc, meta, sel, cu, out, scratch)
                lens = (cu[1:] - cu[:-1]).to(torch.int64)
                o = out.float()
                live_zero = ((o.abs().sum(-1) == 0) & (lens[:, None] > 0)).any()
                bad.bitwise_or_((cnt != 0).any().to(torch.int32))
                bad.bitwise_or_(2 * (~torch.isfinite(o).all()).to(torch.int32))
                bad.bitwise_or_(4 * live_zero.to(torch.int32))
                replay.add_(1)

            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                body()  # warm-up outside capture (kernel attributes, allocator)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            replay.zero_()
            bad.zero_()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                body()
            rng = np.random.default_rng(bs * 131 + hq)
            for r in range(REPLAYS):
                graph.replay()
                if (r + 1) % CHECK_EVERY == 0 or r == 0:
                    torch.cuda.synchronize()
                    # host regeneration of this replay's inputs
                    hsel = torch.zeros(bs * cap, dtype=torch.int32)
                    hcu = torch.zeros(bs + 1, dtype=torch.int32)
                    I.replay_inputs(SEED, torch.tensor([r]), bs, band, cap, SLOTS, hsel, hcu)
                    assert torch.equal(hcu, cu.cpu()), "device and host regeneration differ"
                    rows = sorted(set(rng.integers(0, bs, size=min(2, bs)).tolist()))
                    ref = oracle.decode(q.cpu(), k_host, v_host, "bf16", hsel, hcu, 1 / 16,
                                        rows=rows)
                    got = out[rows].float().cpu().double().numpy()
                    err = rel_l2(got, oracle.round_bf16(ref))
                    assert err.max() <= REL_L2_TOL, (hq, band, bs, r, err.max())
                    worst = max(worst, float(err.max()))
            torch.cuda.synchronize()
            assert int(bad.item()) == 0, (hq, band, bs, int(bad.item()))
            assert int(replay.item()) == REPLAYS
            assert qsa.qsa_scratch_error(scratch) == 0
            del graph
    return worst


@pytest.mark.parametrize("hq", [24, 12])
def test_graph_replay_sweep(cuda_device, hq):
    worst = _sweep_topology(cuda_device, hq)
    print(f"Hq={hq}: worst rel-L2 over checked replays {worst:.3e}")


def test_counter_stress_150k_launches(cuda_device):
    """bs=17 TP1 long selections split across CTAs; 150,000 launches; counters zero."""
    g = torch.Generator().manual_seed(17)
    lengths = torch.randint(1500, 2056, (17,), generator=g)
    w = I.tp1_mixed(seed=17, bs=17, num_slots=65536, lengths=lengths).to(cuda_device)
    out0 = torch.empty_like(w.q)
    out = torch.empty_like(w.q)
    scratch = qsa.alloc_scratch(w.bs, w.num_q_heads, w.capacity, cuda_device)
    meta = qsa.KVQuantMeta("bf16", w.capacity, None, None, w.softmax_scale)
    assert qsa.qsa_decode_grid(w.bs, w.num_q_heads, w.capacity) > 1
    qsa.qsa_decode(w.q, w.k_pool, w.v_pool, meta, w.sel, w.cu, out0, scratch)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(100):
            qsa.qsa_decode(w.q, w.k_pool, w.v_pool, meta, w.sel, w.cu, out, scratch)
    for _ in range(1500):
        graph.replay()
    torch.cuda.synchronize()
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    assert qsa.qsa_scratch_error(scratch) == 0
    assert torch.equal(out, out0)
