"""A decode step as a server runs it: the KV write of the step's new tokens
followed by the decode over selections that include them, captured once in a
CUDA graph and replayed with new token values (sglang PR #36845, "Changes":
captured graphs replay without host readback; sglang PR #37798,
"Modifications": the write is one fused quantise + scatter launch). Sampled
replays are compared with the oracle's write and decode of the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, counters, meta_for, run_oracle

pytestmark = pytest.mark.gpu

BS, SLOTS, REPLAYS = 8, 16384, 40


def _host_pools(w):
    """numpy copies of a tiered workload's pools, for oracle.write_tiered."""
    d = {"k_pool": w.k_pool, "v_pool": w.v_pool, "k_scale": w.k_scale, "v_scale": w.v_scale}
    d.update({k: w.extra[k] for k in I.TIER_KEYS})
    return {k: v.cpu().numpy().copy() for k, v in d.items()}


@pytest.mark.parametrize("fmt", ["int8", "int4_g32", I.TIERED])
def test_write_then_decode_step_replayed_in_a_graph(cuda_device, fmt):
    dev = cuda_device
    g = torch.Generator().manual_seed(70)
    lengths = [1, 64, 700, 2055, 33, 1200, 9, 400]
    if fmt == I.TIERED:
        w = I.tiered(seed=71, bs=BS, num_slots=SLOTS, ring_slots=1024, lengths=lengths)
    else:
        w = I.tp1_mixed(seed=71, bs=BS, num_slots=SLOTS, lengths=lengths, fmt=fmt)
    # each sequence's newest token goes to a fresh slot, which its selection includes
    new_slots = torch.randperm(SLOTS, generator=g)[:BS].to(torch.int32)
    cu = w.cu.long()
    for b in range(BS):
        w.sel[cu[b + 1] - 1] = new_slots[b]
    wd = w.to(dev)
    xk = torch.zeros(BS, 2, 256, dtype=torch.bfloat16, device=dev)
    xv = torch.zeros_like(xk)
    slots_d = new_slots.to(dev)
    out = torch.zeros_like(wd.q)
    scratch = qsa.alloc_scratch(BS, 24, wd.capacity, dev)
    meta = meta_for(wd)
    tier = {k: wd.extra[k] for k in I.TIER_KEYS} if fmt == I.TIERED else None

    def step():
        if tier is not None:
            qsa.qsa_kv_write_tiered(xk, xv, slots_d, wd.k_pool, wd.v_pool, wd.k_scale, wd.v_scale, tier)
        else:
            qsa.qsa_kv_write(fmt, xk, xv, slots_d, wd.k_pool, wd.v_pool, wd.k_scale, wd.v_scale)
        qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta, wd.sel, wd.cu, out, scratch)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    host = None
    for r in range(REPLAYS):
        hk = I.normal_values((BS, 2, 256), 1000 + r).to(torch.bfloat16)
        hv = I.normal_values((BS, 2, 256), 2000 + r, std=0.5).to(torch.bfloat16)
        xk.copy_(hk)
        xv.copy_(hv)
        graph.replay()
        if r % 13 == 0 or r == REPLAYS - 1:
            torch.cuda.synchronize()
            # the oracle writes the same rows into host copies of the pools, then decodes
            if fmt == I.TIERED:
                hp = _host_pools(wd)
                # the pools already hold this replay's write; the oracle's write of the
                # same tokens over a copy of them must change nothing (every written
                # row, scale and owner is the oracle's), then decode from the pools
                ref_pools = {k: v.copy() for k, v in hp.items()}
                oracle.write_tiered(hk, hv, new_slots, ref_pools)
                for k in hp:
                    assert np.array_equal(ref_pools[k].view(np.uint8), hp[k].view(np.uint8)), (r, k)
                host = I.Workload(w.q, torch.from_numpy(hp["k_pool"]), torch.from_numpy(hp["v_pool"]),
                                  w.sel, w.cu, fmt, torch.from_numpy(hp["k_scale"]),
                                  torch.from_numpy(hp["v_scale"]), w.softmax_scale, w.capacity,
                                  extra={k: torch.from_numpy(hp[k]) for k in I.TIER_KEYS})
            else:
                for x, pool, sc in ((hk, wd.k_pool, wd.k_scale), (hv, wd.v_pool, wd.v_scale)):
                    codes, scales = oracle.quantize_rows(x.reshape(BS * 2, 256), fmt)
                    got = pool.cpu()[new_slots.long()].reshape(BS * 2, -1).view(torch.uint8).numpy()
                    assert np.array_equal(got, codes.view(np.uint8)), r
                    gs = sc.cpu()[new_slots.long()].reshape(BS * 2, -1).numpy()
                    assert np.array_equal(gs.view(np.uint8), np.asarray(scales).reshape(BS * 2, -1).view(np.uint8)), r
                host = I.Workload(w.q, wd.k_pool.cpu(), wd.v_pool.cpu(), w.sel, w.cu, fmt,
                                  wd.k_scale.cpu(), wd.v_scale.cpu(), w.softmax_scale, w.capacity)
            compare(out, run_oracle(host), np.asarray(lengths))
            assert (counters(scratch, BS, 24, wd.capacity) == 0).all()
    assert qsa.qsa_scratch_error(scratch) == 0
    del graph
