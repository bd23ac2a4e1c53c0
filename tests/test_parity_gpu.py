"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Every comparison is per (sequence, head) relative L2 over the 256 output
dims, against the oracle rounded to bf16, with a 2e-3 bound.
"""
import numpy as np
import pytest
import torch

import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, counters, gather_subset, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


def _parity(w, dev, max_ctas=0):
    wd = w.to(dev)
    out, scratch = run_cuda(wd, max_ctas)
    torch.cuda.synchronize()
    ref = run_oracle(w)
    eb, eu = compare(out, ref, w.lengths().numpy())
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    return out, eb, eu


@pytest.mark.parametrize("fmt", I.FORMATS)
@pytest.mark.parametrize("length", [1, 31, 32, 33, 64, 77, 2055])
def test_tiny_tp2(cuda_device, fmt, length):
    w = I.tiny_tp2(seed=0, length=length, fmt=fmt)
    _parity(w, cuda_device)


@pytest.mark.parametrize("fmt", I.FORMATS)
def test_tp1_mixed_lengths(cuda_device, fmt):
    w = I.tp1_mixed(seed=1, bs=16, fmt=fmt)
    _parity(w, cuda_device)


@pytest.mark.parametrize("max_ctas", [1, 2, 3, 7, 0])
def test_split_count_invariance(cuda_device, max_ctas):
    """Forcing one CTA (no split) or several gives the same answer within rounding."""
    w = I.tp1_mixed(seed=5, bs=6, num_slots=8192, lengths=[2055, 1, 700, 0, 64, 1500])
    out, _, _ = _parity(w, cuda_device, max_ctas)
    wd = w.to(cuda_device)
    base, _ = run_cuda(wd, 1)
    torch.cuda.synchronize()
    a = out.float().cpu().double().numpy()
    b = base.float().cpu().double().numpy()
    num = np.sqrt(((a - b) ** 2).sum(-1))
    den = np.sqrt((b ** 2).sum(-1))
    live = den > 0
    # both are bf16 roundings of nearly equal FP32 results: at most isolated 1-ulp flips
    assert (num[live] / den[live]).max() <= 2e-3


def test_edge_lengths_and_empty_rows(cuda_device):
    lengths = [0, 1, 2055, 0, 5, 64, 65, 0, 33, 2054]
    w = I.tp1_mixed(seed=6, bs=len(lengths), num_slots=16384, lengths=lengths)
    _parity(w, cuda_device)


def test_all_empty(cuda_device):
    w = I.tp1_mixed(seed=6, bs=4, num_slots=1024, lengths=[0, 0, 0, 0])
    w.capacity = 16
    wd = w.to(cuda_device)
    out, scratch = run_cuda(wd)
    torch.cuda.synchronize()
    assert (out == 0).all()
    assert qsa.qsa_scratch_error(scratch) == 0


def test_single_index_is_bitwise_the_v_row(cuda_device):
    w = I.tp1_mixed(seed=7, bs=32, num_slots=4096, lengths=[1] * 32)
    wd = w.to(cuda_device)
    out, _ = run_cuda(wd)
    torch.cuda.synchronize()
    ref = torch.stack([w.v_pool[int(w.sel[b])].repeat_interleave(12, 0) for b in range(32)])
    assert torch.equal(out.cpu(), ref)


def test_duplicates_only(cuda_device):
    """A selection of one slot repeated n times equals that slot's V row."""
    w = I.tp1_mixed(seed=8, bs=3, num_slots=4096, lengths=[5, 300, 2055])
    w.sel[:] = 1234
    wd = w.to(cuda_device)
    out, _ = run_cuda(wd)
    torch.cuda.synchronize()
    ref = w.v_pool[1234].repeat_interleave(12, 0)
    for b in range(3):
        assert torch.equal(out[b].cpu(), ref)


def test_bs128_tiny_lengths(cuda_device):
    g = torch.Generator().manual_seed(9)
    lengths = torch.randint(0, 4, (128,), generator=g)
    w = I.tp1_mixed(seed=9, bs=128, num_slots=4096, lengths=lengths)
    _parity(w, cuda_device)


def test_repeat_launches_deterministic_and_counters_reset(cuda_device):
    w = I.tp1_mixed(seed=10, bs=17, num_slots=65536, max_len=2055)
    wd = w.to(cuda_device)
    out0, scratch = run_cuda(wd)
    outs = torch.empty_like(out0)
    for _ in range(200):
        run_cuda(wd, out=outs, scratch=scratch)
    torch.cuda.synchronize()
    assert torch.equal(out0, outs)
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    assert qsa.qsa_scratch_error(scratch) == 0


def test_device_error_flags(cuda_device):
    w = I.tp1_mixed(seed=11, bs=4, num_slots=2048, lengths=[10, 20, 30, 40])
    wd = w.to(cuda_device)
    bad = wd.sel.clone()
    bad[15] = w.num_slots + 5
    bad[16] = -3
    out = torch.empty_like(wd.q)
    scratch = qsa.alloc_scratch(w.bs, w.num_q_heads, w.capacity, cuda_device)
    meta = qsa.KVQuantMeta("bf16", w.capacity, None, None, w.softmax_scale)
    qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta, bad, wd.cu, out, scratch)
    assert qsa.qsa_scratch_error(scratch, clear=True) == qsa.binding.DEVERR_SLOT_RANGE
    assert qsa.qsa_scratch_error(scratch) == 0
    # decreasing cu_seqlens and a length above capacity
    cu = wd.cu.clone()
    cu[2] = cu[1] - 1
    qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta, wd.sel, cu, out, scratch)
    assert qsa.qsa_scratch_error(scratch, clear=True) & qsa.binding.DEVERR_CU_SEQLENS
    meta_small = qsa.KVQuantMeta("bf16", 25, None, None, w.softmax_scale)
    qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta_small, wd.sel, wd.cu, out, scratch)
    assert qsa.qsa_scratch_error(scratch, clear=True) & qsa.binding.DEVERR_CU_SEQLENS
    # the library keeps working afterwards
    out2, _ = run_cuda(wd, scratch=scratch)
    torch.cuda.synchronize()
    compare(out2, run_oracle(w), w.lengths().numpy())
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()


def test_strided_q_and_out(cuda_device):
    """q and out may be views with padded batch/head strides."""
    w = I.tp1_mixed(seed=12, bs=5, num_slots=4096, lengths=[3, 100, 2055, 40, 1])
    wd = w.to(cuda_device)
    qbig = torch.zeros(5, 30, 264, dtype=torch.bfloat16, device=cuda_device)
    qv = qbig[:, 3:27, 8:]
    qv.copy_(wd.q)
    obig = torch.zeros(5, 26, 272, dtype=torch.bfloat16, device=cuda_device)
    ov = obig[:, 1:25, 16:]
    wd.q = qv
    run_cuda(wd, out=ov)
    torch.cuda.synchronize()
    compare(ov, run_oracle(w), w.lengths().numpy())
    assert (obig[:, 0] == 0).all() and (obig[:, :, :16] == 0).all()


@pytest.mark.parametrize("fmt", I.FORMATS)
def test_headline_saturated_sampled(cuda_device, fmt):
    """bs=128, L=2055, 24Q/2KV over a 1M-slot pool: sampled sequences vs the oracle."""
    w = I.tp1_saturated(seed=2, device=cuda_device, fmt=fmt)
    out, scratch = run_cuda(w)
    torch.cuda.synchronize()
    rows = [0, 1, 37, 64, 100, 127]
    sub = gather_subset(w, rows)
    ref = run_oracle(sub)
    compare(out[rows], ref, [2055] * len(rows))
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    # every row is finite and non-degenerate
    o = out.float()
    assert torch.isfinite(o).all() and (o.abs().sum(-1) > 0).all()


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "int8", "int4", "int8_g64", "int4_g32"])
def test_every_code_dequantises_exactly(cuda_device, fmt):
    """A single selected slot whose V row holds every code of the format, with a
    unit scale: the output row is exactly the decoded codes (NaN codes give NaN)."""
    w = I.tiny_tp2(seed=40, length=1, fmt=fmt)
    slot = int(w.sel[0])
    if fmt in ("int4", "int4_g32"):
        codes = torch.arange(256, dtype=torch.int32) % 16
        row = (codes[0::2] | (codes[1::2] << 4)).to(torch.uint8)
        if fmt == "int4":
            vals = torch.where(codes >= 8, codes - 16, codes).float()
        else:
            vals = (codes - 8).float()        # offset binary
    elif fmt in ("int8", "int8_g64"):
        row = torch.arange(-128, 128, dtype=torch.int32).to(torch.int8)
        vals = row.float()
    else:
        row = torch.arange(256, dtype=torch.int32).to(torch.uint8)
        vals = row.view(torch.float8_e4m3fn).float()
    w.v_pool[slot, 0] = row
    w.v_scale = torch.ones_like(w.v_scale)
    wd = w.to(cuda_device)
    out, _ = run_cuda(wd)
    torch.cuda.synchronize()
    ref = vals.to(torch.bfloat16).float()
    got = out[0].float().cpu()
    for h in range(12):
        nan = torch.isnan(ref)
        assert torch.equal(torch.isnan(got[h]), nan)
        assert torch.equal(got[h][~nan], ref[~nan])


@pytest.mark.parametrize("fmt", ["int8_g64", "int4_g32"])
def test_group_scales_reach_their_channels(cuda_device, fmt):
    """One selected slot, V codes all 1 (int4_g32: nibble 9), V scale of group k
    = 2^k: output channel d reads exactly the scale of its group."""
    w = I.tiny_tp2(seed=41, length=1, fmt=fmt)
    slot = int(w.sel[0])
    G = I.HEAD_DIM // I.GROUPED[fmt]
    w.v_pool[slot, 0] = 0x99 if fmt == "int4_g32" else 1
    w.v_scale[slot, 0] = torch.tensor([2.0 ** k for k in range(G)], dtype=torch.float16)
    wd = w.to(cuda_device)
    out, _ = run_cuda(wd)
    torch.cuda.synchronize()
    ref = torch.tensor([2.0 ** (d // I.GROUPED[fmt]) for d in range(256)])
    for h in range(12):
        assert torch.equal(out[0, h].float().cpu(), ref)


@pytest.mark.parametrize("max_ctas", [0, 1])
def test_int8_wide_v_scales(cuda_device, max_ctas):
    """int8 PV runs in f16 on P * s_v * 2^-E_h with a per-head offset E_h that must
    follow the largest products: per-slot V scales spread over 2^-40 .. 2^40, and
    along one selection rising from 2^-30 to 2^30 (the offset rises stage after
    stage), against the oracle, with the split merge (all CTAs) and without (one)."""
    lengths = [2055, 700, 64, 1, 1500, 300]
    w = I.tp1_mixed(seed=71, bs=len(lengths), num_slots=8192, fmt="int8", lengths=lengths)
    g = torch.Generator().manual_seed(71)
    vs = w.v_scale.double().clone()
    vs *= torch.pow(2.0, torch.randint(-40, 41, vs.shape, generator=g).double())
    lo, hi = int(w.cu[4]), int(w.cu[5])
    ramp = torch.pow(2.0, torch.linspace(-30.0, 30.0, hi - lo, dtype=torch.float64))
    vs[w.sel[lo:hi].long()] = w.v_scale.double()[w.sel[lo:hi].long()] * ramp[:, None]
    w.v_scale = vs.float()
    _parity(w, cuda_device, max_ctas)


def _equal_lengths(seed, hq, bs, length, num_slots=65536):
    hkv = hq // 12
    kc, vc, ks, vs = I.make_pools(num_slots, hkv, "bf16", seed)
    g = torch.Generator().manual_seed(seed)
    sel = I.uniform_indices(bs * length, num_slots, g)
    return I.Workload(I.make_query(bs, hq, seed), kc, vc, sel, I.cu_from_lengths([length] * bs),
                      "bf16", ks, vs, capacity=length, name=f"equal_{hq}q_bs{bs}_L{length}")


@pytest.mark.parametrize("hq,bs,length", [
    (24, 1, 2055), (24, 3, 777), (24, 5, 2055), (24, 8, 2055), (24, 12, 700), (24, 20, 600),
    (24, 32, 500), (12, 7, 1000), (12, 13, 333),
])
def test_equal_length_splits_every_fan_in(cuda_device, hq, bs, length):
    """Equal lengths, a whole number of CTAs per (sequence, KV head) segment (fan-ins
    16, 12, 15, 9, 6, 3, 2, 15 and 5 here): every contributor merges a slice of its
    segment from all partials; the output, the error word and the counters."""
    w = _equal_lengths(80 + bs, hq, bs, length)
    out, scratch = run_cuda(w.to(cuda_device))
    torch.cuda.synchronize()
    compare(out, run_oracle(w), w.lengths().numpy())
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    again, _ = run_cuda(w.to(cuda_device), scratch=scratch)
    torch.cuda.synchronize()
    assert torch.equal(again, out)


def _given_lengths(seed, hq, lengths, num_slots=65536):
    hkv = hq // 12
    kc, vc, ks, vs = I.make_pools(num_slots, hkv, "bf16", seed)
    g = torch.Generator().manual_seed(seed)
    sel = I.uniform_indices(int(sum(lengths)), num_slots, g)
    return I.Workload(I.make_query(len(lengths), hq, seed), kc, vc, sel, I.cu_from_lengths(lengths),
                      "bf16", ks, vs, capacity=max(lengths), name=f"given_{hq}q_bs{len(lengths)}")


@pytest.mark.parametrize("hq,lengths", [
    (24, [2055, 100]),                       # few segments, each split into its own CTAs
    (12, [700, 65, 2055, 300]),
    (12, [2055, 5, 700]),                    # a selection shorter than the CTAs per segment
    (24, [1500, 1400, 1300, 1450, 1350]),    # ten nearly equal segments
])
def test_small_batches_of_unequal_lengths(cuda_device, hq, lengths):
    w = _given_lengths(90 + len(lengths), hq, lengths)
    out, scratch = run_cuda(w.to(cuda_device))
    torch.cuda.synchronize()
    compare(out, run_oracle(w), w.lengths().numpy())
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    again, _ = run_cuda(w.to(cuda_device), scratch=scratch)
    torch.cuda.synchronize()
    assert torch.equal(again, out)
