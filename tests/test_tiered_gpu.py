"""GPU parity of the tiered int8ring_int4 pool (sglang PR #37798, "Modifications",
the tiered KV pool module): the decode reads the int8_g64 ring row of a slot whose
ring position it owns and the int4_g32 row otherwise; the write stores both and
stamps the owner, the last token of a write taking a shared ring position."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import binding as B
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, counters, gather_subset, rel_l2, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


def _parity(w, dev):
    wd = w.to(dev)
    out, scratch = run_cuda(wd)
    torch.cuda.synchronize()
    compare(out, run_oracle(w), w.lengths().numpy())
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    return out


def _within_one_ulp(a, b):
    """The tiered kernel widens its cold int4 rows into int8 tiles and runs the
    int8 fragment path over them, the int4-g32 kernel unpacks nibbles straight
    into its fragments: the same products, summed in another order inside the
    MMAs. An output may then differ by one bf16 ulp at its (sequence, head)
    row's scale (an output near zero is a cancelling sum), and rarely."""
    a, b = a.float(), b.float()
    d = (a - b).abs()
    row = torch.maximum(a.abs(), b.abs()).amax(dim=-1, keepdim=True)
    _, e = torch.frexp(row)
    ulp = torch.ldexp(torch.ones_like(row), e - 8)  # bf16: 8 significant bits
    assert bool((d <= ulp).all()), float((d / ulp).max())
    ndiff = int((d > 0).sum())
    assert ndiff <= max(4, a.numel() // 1000), ndiff


@pytest.mark.parametrize("hot_share", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("ring", [1024, 4096])
def test_tiered_parity(cuda_device, hot_share, ring):
    w = I.tiered(seed=50, bs=8, num_slots=16384, ring_slots=ring, hot_share=hot_share,
                 lengths=[1, 33, 64, 700, 2055, 5, 1500, 0])
    _parity(w, cuda_device)


def test_tiered_tp2(cuda_device):
    w = I.tiered(seed=51, bs=3, num_slots=8192, ring_slots=2048, num_kv_heads=1,
                 lengths=[2055, 77, 1])
    _parity(w, cuda_device)


def test_all_cold_matches_the_int4_g32_kernel_and_all_hot_the_oracle_int8_g64(cuda_device):
    w = I.tiered(seed=52, bs=6, num_slots=8192, ring_slots=8192, lengths=[64, 2055, 9, 512, 1, 300])
    cold = I.Workload(w.q, w.k_pool, w.v_pool, w.sel, w.cu, w.fmt, w.k_scale, w.v_scale,
                      capacity=w.capacity, extra=dict(w.extra))
    cold.extra["owner"] = torch.full_like(w.extra["owner"], -1)
    out_t, _ = run_cuda(cold.to(cuda_device))
    g32 = I.Workload(w.q, w.k_pool, w.v_pool, w.sel, w.cu, "int4_g32", w.k_scale, w.v_scale,
                     capacity=w.capacity)
    out_4, _ = run_cuda(g32.to(cuda_device))
    torch.cuda.synchronize()
    _within_one_ulp(out_t, out_4)
    # all hot: the ring has one row per slot (R = num_slots) and owner[p] = p
    hot = I.Workload(w.q, w.k_pool, w.v_pool, w.sel, w.cu, w.fmt, w.k_scale, w.v_scale,
                     capacity=w.capacity, extra=dict(w.extra))
    hot.extra["owner"] = torch.arange(8192, dtype=torch.int32)
    t = w.extra
    ring_ids = torch.arange(8192)
    xk = I.normal_values((8192, 2, 256), 53)
    hot.extra["k_ring"], hot.extra["k_ring_scale"] = I.quantize_pool(xk, "int8_g64")
    xv = I.normal_values((8192, 2, 256), 54)
    hot.extra["v_ring"], hot.extra["v_ring_scale"] = I.quantize_pool(xv, "int8_g64")
    out_h, _ = run_cuda(hot.to(cuda_device))
    torch.cuda.synchronize()
    ref = oracle.decode(w.q, hot.extra["k_ring"], hot.extra["v_ring"], "int8_g64", w.sel, w.cu,
                        w.softmax_scale, hot.extra["k_ring_scale"], hot.extra["v_ring_scale"])
    compare(out_h, ref, w.lengths().numpy())
    assert ring_ids.numel() == t["owner"].numel()


@pytest.mark.parametrize("seed,lengths", [
    (60, [2055]),                      # two segments of 16 CTAs each
    (61, [2055, 2055]),
    (62, [2055] * 4),
    (63, [2055, 1500, 700]),           # unequal: the equal-token split
    (64, [2055] * 16),
    (65, [1, 2055, 33, 2055, 64]),
])
def test_all_cold_matches_the_int4_g32_kernel_at_any_split(cuda_device, seed, lengths):
    """Segments cut into many pieces: an all-cold tiered call meets the oracle's
    gate and stays within one bf16 ulp of the int4-g32 call."""
    w = I.tiered(seed=seed, bs=len(lengths), num_slots=8192, ring_slots=2048, lengths=lengths)
    cold = I.Workload(w.q, w.k_pool, w.v_pool, w.sel, w.cu, w.fmt, w.k_scale, w.v_scale,
                      capacity=w.capacity, extra=dict(w.extra))
    cold.extra["owner"] = torch.full_like(w.extra["owner"], -1)
    g32 = I.Workload(w.q, w.k_pool, w.v_pool, w.sel, w.cu, "int4_g32", w.k_scale, w.v_scale,
                     capacity=w.capacity)
    out_t, _ = run_cuda(cold.to(cuda_device))
    out_4, _ = run_cuda(g32.to(cuda_device))
    torch.cuda.synchronize()
    _within_one_ulp(out_t, out_4)
    compare(out_t, run_oracle(g32), w.lengths().numpy())


def test_tiered_headline_sampled(cuda_device):
    """bs=128, L=2055, 24Q/2KV over a 1M-slot pool with the pages' 8192-row ring,
    a quarter of each selection hot: sampled sequences against the oracle."""
    pools = I.make_tiered_pools(1048576, 2, I.RING_SLOTS, 55, device=cuda_device)
    w = I.tiered(seed=55, device=cuda_device, bs=128, num_slots=1048576, ring_slots=I.RING_SLOTS,
                 lengths=[2055] * 128, hot_share=0.25, pools=pools)
    assert w.q.is_cuda and w.sel.is_cuda and w.cu.is_cuda
    out, scratch = run_cuda(w)
    torch.cuda.synchronize()
    rows = [0, 1, 63, 127]
    sub = gather_subset(w, rows)
    compare(out[rows], run_oracle(sub), [2055] * len(rows))
    assert qsa.qsa_scratch_error(scratch) == 0
    assert torch.isfinite(out.float()).all()


def _tier_buffers(slots, R, hkv, dev, g):
    bufs = {
        "k_pool": torch.randint(0, 256, (slots, hkv, 128), generator=g, dtype=torch.int32).to(torch.uint8),
        "v_pool": torch.randint(0, 256, (slots, hkv, 128), generator=g, dtype=torch.int32).to(torch.uint8),
        "k_scale": torch.full((slots, hkv, 8), 3.0, dtype=torch.float16),
        "v_scale": torch.full((slots, hkv, 8), 5.0, dtype=torch.float16),
        "k_ring": torch.randint(-128, 128, (R, hkv, 256), generator=g, dtype=torch.int32).to(torch.int8),
        "v_ring": torch.randint(-128, 128, (R, hkv, 256), generator=g, dtype=torch.int32).to(torch.int8),
        "k_ring_scale": torch.full((R, hkv, 4), 7.0, dtype=torch.float16),
        "v_ring_scale": torch.full((R, hkv, 4), 11.0, dtype=torch.float16),
        "owner": torch.randint(-1, slots, (R,), generator=g).to(torch.int32),
    }
    return bufs, {k: v.to(dev) for k, v in bufs.items()}


def _write_tiered_gpu(dev_bufs, xk, xv, sl, err=None):
    qsa.qsa_kv_write_tiered(xk, xv, sl, dev_bufs["k_pool"], dev_bufs["v_pool"], dev_bufs["k_scale"],
                            dev_bufs["v_scale"], {k: dev_bufs[k] for k in I.TIER_KEYS}, err)


@pytest.mark.parametrize("hkv", [2, 1])
def test_tiered_write_matches_the_oracle_with_ring_wrap_and_collisions(cuda_device, hkv):
    """R = 64 over 4096 slots (the pages' ring-wrap test), 500 tokens per write: pools,
    ring rows, scales and owners bit-equal to the oracle's in-order write; the same
    write repeated 20 times gives the same bytes."""
    slots, R, n = 4096, 64, 500
    g = torch.Generator().manual_seed(56)
    host, dev = _tier_buffers(slots, R, hkv, cuda_device, g)
    sl = torch.randperm(slots, generator=g)[:n].to(torch.int32)
    xk = I.normal_values((n, hkv, 256), 57, std=2.0).to(torch.bfloat16)
    xv = I.normal_values((n, hkv, 256), 58, std=0.5).to(torch.bfloat16)
    xk[3] = 0.0
    ref = {k: v.numpy().copy() for k, v in host.items()}
    oracle.write_tiered(xk, xv, sl, ref)
    first = None
    for rep in range(20):
        d = {k: v.clone() for k, v in dev.items()}
        err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        _write_tiered_gpu(d, xk.to(cuda_device), xv.to(cuda_device), sl.to(cuda_device), err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = {k: v.cpu() for k, v in d.items()}
        if first is None:
            first = got
            for k in host:
                a = got[k].numpy()
                assert np.array_equal(a.view(np.uint8), ref[k].view(np.uint8)), k
        else:
            for k in host:
                assert torch.equal(got[k], first[k]), (rep, k)


def test_tiered_write_then_decode(cuda_device):
    """Tokens written by qsa_kv_write_tiered decode like the oracle says, hot and cold."""
    w = I.tiered(seed=59, bs=4, num_slots=8192, ring_slots=1024, lengths=[100, 2055, 1, 640])
    wd = w.to(cuda_device)
    fresh = torch.unique(w.sel)[:700]
    n = fresh.numel()
    xk = I.normal_values((n, 2, 256), 60).to(torch.bfloat16)
    xv = I.normal_values((n, 2, 256), 61).to(torch.bfloat16)
    qsa.qsa_kv_write_tiered(xk.to(cuda_device), xv.to(cuda_device), fresh.to(cuda_device),
                            wd.k_pool, wd.v_pool, wd.k_scale, wd.v_scale,
                            {k: wd.extra[k] for k in I.TIER_KEYS})
    out, _ = run_cuda(wd)
    torch.cuda.synchronize()
    host = I.Workload(w.q, wd.k_pool.cpu(), wd.v_pool.cpu(), w.sel, w.cu, w.fmt, wd.k_scale.cpu(),
                      wd.v_scale.cpu(), w.softmax_scale, w.capacity,
                      extra={k: wd.extra[k].cpu() for k in I.TIER_KEYS})
    own = host.extra["owner"]
    hot = (own[(fresh & 1023).long()] == fresh).sum().item()
    assert hot > 0                                   # the write made some rows hot
    compare(out, run_oracle(host), w.lengths().numpy())


def test_tiered_write_flags_bad_slots(cuda_device):
    g = torch.Generator().manual_seed(62)
    host, dev = _tier_buffers(512, 64, 2, cuda_device, g)
    sl = (torch.arange(40, dtype=torch.int32) * 7)
    sl[4] = 600
    sl[9] = -1
    xk = I.normal_values((40, 2, 256), 63).to(torch.bfloat16)
    ref = {k: v.numpy().copy() for k, v in host.items()}
    ok = torch.tensor([i not in (4, 9) for i in range(40)])
    oracle.write_tiered(xk[ok], xk[ok], sl[ok], ref)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    _write_tiered_gpu(dev, xk.to(cuda_device), xk.to(cuda_device), sl.to(cuda_device), err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.DEVERR_SLOT_RANGE
    for k in ("k_pool", "k_scale"):
        assert np.array_equal(dev[k].cpu().numpy().view(np.uint8), ref[k].view(np.uint8)), k
    # the ring rows and owners of the valid tokens' positions follow the in-order rule
    # over the valid tokens (the claim skips bad slots, so token indices shift only
    # in which of them is last -- the same slots win)
    assert np.array_equal(dev["owner"].cpu().numpy(), ref["owner"])
    assert np.array_equal(dev["k_ring"].cpu().numpy(), ref["k_ring"])
