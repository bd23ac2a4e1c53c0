"""GPU parity of the quantising KV write (qsa_kv_write) against the oracle.

Codes and scales are integers / exact binary32 decisions, so the bar is bit
equality with oracle.quantize_rows on the same inputs; rows that are not
written must keep their bytes.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import binding as B
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

ROW = {"bf16": 256, "fp8_e4m3": 256, "int8": 256, "int4": 128, "int8_g64": 256, "int4_g32": 128}
DT = {"bf16": torch.bfloat16, "fp8_e4m3": torch.uint8, "int8": torch.int8, "int4": torch.uint8,
      "int8_g64": torch.int8, "int4_g32": torch.uint8}


def _scales(fmt, slots_n, hkv, dev, fill):
    """Scale buffers of a pool: fp32 per (slot, head), binary16 per group, fp8 [1]."""
    if fmt in I.GROUPED:
        return torch.full((slots_n, hkv, 256 // I.GROUPED[fmt]), fill, dtype=torch.float16, device=dev)
    return torch.full((slots_n, hkv), fill, device=dev)


def _bits(t):
    """Scales as comparable integer bits (float32 or binary16)."""
    a = t.numpy() if hasattr(t, "numpy") else t
    return a.view(np.uint16 if a.dtype == np.float16 else np.uint32).reshape(-1)


def _new_rows(n, hkv, seed):
    g = torch.Generator().manual_seed(seed)
    std = torch.exp(torch.randn(n, hkv, 1, generator=g))
    x = (torch.randn(n, hkv, 256, generator=g) * std).to(torch.bfloat16)
    x[0] = 0.0                                   # all-zero row -> scale 0, zero codes
    x[1] = x[1].float().mul(1000).to(torch.bfloat16)   # fp8 saturation
    tie = torch.zeros(256)
    tie[0] = 127.0
    tie[1:20] = torch.arange(19) + 0.5           # exact halves at scale 1 (int8)
    x[2, 0] = tie.to(torch.bfloat16)
    # bf16 subnormals: the scale leaves the normal range and codes need the clamp
    x[3, 0] = (torch.arange(256) % 200 - 90).float().mul(2.0 ** -133).to(torch.bfloat16)
    # magnitudes near the bf16 maximum
    x[4, 0] = (torch.linspace(-1, 1, 256) * 3.38e38).to(torch.bfloat16)
    # int4 ties: absmax 7 gives scale 1, halves round to even
    tie4 = torch.zeros(256)
    tie4[0] = -7.0
    tie4[1:15] = torch.arange(14) * 0.5 - 3.25 + 0.25
    x[5, 0] = tie4.to(torch.bfloat16)
    # e4m3 midpoints at a power-of-two scale (exact quotients): 1 + 1/16, 2 + 1/8, ...
    mid = torch.tensor([1.0625, 1.1875, 2.125, 3.375, 0.0146484375, 464.0, 0.001953125, -1.0625])
    x[6, 0, :8] = (mid * 0.25).to(torch.bfloat16)
    return x


def _pools(fmt, slots, hkv, dev, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (slots, hkv, ROW[fmt])
    if fmt == "bf16":
        mk = lambda: torch.randn(shape, generator=g).to(torch.bfloat16)
    else:
        mk = lambda: torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(torch.uint8).view(DT[fmt])
    return mk().to(dev), mk().to(dev)


@pytest.mark.parametrize("fp8_scales", [(0.05, 0.02), (0.25, 0.25)])
@pytest.mark.parametrize("hkv", [2, 1])
@pytest.mark.parametrize("fmt", I.FORMATS)
def test_kv_write_matches_oracle(cuda_device, fmt, hkv, fp8_scales):
    if fmt != "fp8_e4m3" and fp8_scales != (0.05, 0.02):
        pytest.skip("the fp8 scale only matters for the fp8 pool")
    n, slots_n = 1000, 8192
    x_k, x_v = _new_rows(n, hkv, 50), _new_rows(n, hkv, 51)
    slots = torch.randperm(slots_n, generator=torch.Generator().manual_seed(52))[:n].to(torch.int32)
    kp, vp = _pools(fmt, slots_n, hkv, cuda_device, 53)
    kp0, vp0 = kp.clone(), vp.clone()
    ks = vs = None
    if fmt == "fp8_e4m3":
        ks = torch.tensor([fp8_scales[0]], device=cuda_device)
        vs = torch.tensor([fp8_scales[1]], device=cuda_device)
    elif fmt != "bf16":
        ks = _scales(fmt, slots_n, hkv, cuda_device, -1.0)
        vs = _scales(fmt, slots_n, hkv, cuda_device, -1.0)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    qsa.qsa_kv_write(fmt, x_k.to(cuda_device), x_v.to(cuda_device), slots.to(cuda_device),
                     kp, vp, ks, vs, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    written = torch.zeros(slots_n, dtype=torch.bool)
    written[slots.long()] = True
    for x, pool, pool0, sc, fp8s in ((x_k, kp, kp0, ks, fp8_scales[0]),
                                     (x_v, vp, vp0, vs, fp8_scales[1])):
        codes, scales = oracle.quantize_rows(x.reshape(n * hkv, 256), fmt, fp8_scale=fp8s)
        got = pool.cpu()[slots.long()].reshape(n * hkv, -1)
        if fmt == "bf16":
            assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), codes)
        else:
            assert np.array_equal(got.view(torch.uint8).numpy(), codes.view(np.uint8))
        if scales is not None:
            assert np.array_equal(_bits(sc.cpu()[slots.long()]), _bits(scales))
            assert (sc.cpu()[~written] == -1.0).all()
        assert torch.equal(pool.cpu()[~written], pool0.cpu()[~written])


def test_kv_write_flags_bad_slots_and_keeps_going(cuda_device):
    n, slots_n = 64, 512
    x = _new_rows(n, 2, 60).to(cuda_device)
    slots = torch.arange(n, dtype=torch.int32) * 3
    slots[5] = slots_n + 1
    slots[9] = -2
    kp, vp = _pools("int8", slots_n, 2, cuda_device, 61)
    ks = torch.zeros(slots_n, 2, device=cuda_device)
    vs = torch.zeros(slots_n, 2, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    qsa.qsa_kv_write("int8", x, x, slots.to(cuda_device), kp, vp, ks, vs, err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.DEVERR_SLOT_RANGE
    codes, _ = oracle.quantize_rows(x.cpu().reshape(n * 2, 256), "int8")
    ok = [i for i in range(n) if i not in (5, 9)]
    got = kp.cpu()[slots[ok].long()].reshape(len(ok) * 2, 256)
    want = codes.reshape(n, 2, 256)[ok].reshape(len(ok) * 2, 256)
    assert np.array_equal(got.numpy(), want)


def test_kv_write_strided_input(cuda_device):
    n, slots_n = 100, 1024
    big = torch.randn(n, 3, 264, dtype=torch.float32).to(torch.bfloat16).to(cuda_device)
    xv = big[:, 1:3, 8:]
    slots = torch.randperm(slots_n)[:n].to(torch.int32).to(cuda_device)
    kp, vp = _pools("int4", slots_n, 2, cuda_device, 62)
    ks = torch.zeros(slots_n, 2, device=cuda_device)
    vs = torch.zeros(slots_n, 2, device=cuda_device)
    qsa.qsa_kv_write("int4", xv, xv, slots, kp, vp, ks, vs)
    torch.cuda.synchronize()
    codes, scales = oracle.quantize_rows(xv.cpu().contiguous().reshape(n * 2, 256), "int4")
    assert np.array_equal(kp.cpu()[slots.cpu().long()].reshape(n * 2, 128).numpy(), codes)
    assert np.array_equal(ks.cpu()[slots.cpu().long()].reshape(-1).numpy(), scales)


@pytest.mark.parametrize("fmt", ["int8", "fp8_e4m3", "int4", "int8_g64", "int4_g32"])
def test_write_then_decode(cuda_device, fmt):
    """Rows written by qsa_kv_write decode like the oracle says they should."""
    w = I.tp1_mixed(seed=63, bs=4, num_slots=4096, lengths=[100, 2055, 1, 640], fmt=fmt)
    wd = w.to(cuda_device)
    fresh = torch.unique(w.sel)[:300]
    xk, xv = _new_rows(fresh.numel(), 2, 64), _new_rows(fresh.numel(), 2, 65)
    qsa.qsa_kv_write(fmt, xk.to(cuda_device), xv.to(cuda_device), fresh.to(cuda_device),
                     wd.k_pool, wd.v_pool, wd.k_scale, wd.v_scale)
    out, _ = run_cuda(wd)
    torch.cuda.synchronize()
    host = I.Workload(w.q, wd.k_pool.cpu(), wd.v_pool.cpu(), w.sel, w.cu, fmt,
                      None if wd.k_scale is None else wd.k_scale.cpu(),
                      None if wd.v_scale is None else wd.v_scale.cpu(), w.softmax_scale, w.capacity)
    compare(out, run_oracle(host), w.lengths().numpy())


def _ratio_rows(exponent: int, gs: int = 256) -> torch.Tensor:
    """Rows whose every scale group (gs channels) has absmax a = (1 + t/128) 2^exponent
    in its first channel, t taking every bf16 mantissa, and whose other values are
    every bf16 x with 2^-11 a <= |x| <= a (both signs): every ratio x / a that can give
    a nonzero code, so the rounding of every such x / s is checked."""
    per = gs - 1
    rows = []
    for t in range(128):
        a = (1 + t / 128) * 2.0 ** exponent
        xs = [m / 128 * 2.0 ** (exponent + e) for e in range(0, -12, -1) for m in range(128, 256)]
        xs = [v for v in xs if v <= a]
        xs = torch.tensor(xs + [-v for v in xs], dtype=torch.float64)
        groups = [xs[k:k + per] for k in range(0, xs.numel(), per)]
        for r0 in range(0, len(groups), 256 // gs):
            row = torch.zeros(256, dtype=torch.float64)
            for j, chunk in enumerate(groups[r0:r0 + 256 // gs]):
                row[j * gs] = a
                row[j * gs + 1:j * gs + 1 + chunk.numel()] = chunk
            rows.append(row)
    return torch.stack(rows).to(torch.bfloat16)


def _write_and_compare(dev, fmt, x, fp8_scale=None):
    n = x.shape[0]
    xk = x.reshape(n, 1, 256)
    slots = torch.arange(n, dtype=torch.int32)
    kp, vp = _pools(fmt, n, 1, dev, 70)
    if fmt == "fp8_e4m3":
        ks = torch.tensor([fp8_scale], device=dev)
        vs = ks.clone()
    else:
        ks = _scales(fmt, n, 1, dev, 0.0)
        vs = _scales(fmt, n, 1, dev, 0.0)
    xd = xk.to(dev)
    qsa.qsa_kv_write(fmt, xd, xd, slots.to(dev), kp, vp, ks, vs)
    torch.cuda.synchronize()
    codes, scales = oracle.quantize_rows(x, fmt, fp8_scale=1.0 if fp8_scale is None else fp8_scale)
    for pool, sc in ((kp, ks), (vp, vs)):
        got = pool.cpu().reshape(n, -1).view(torch.uint8).numpy()
        assert np.array_equal(got, codes.view(np.uint8)), (fmt, fp8_scale)
        if scales is not None:
            assert np.array_equal(_bits(sc.cpu()), _bits(scales))


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_every_quotient_rounds_like_the_oracle(cuda_device, fmt):
    """All reachable (x, absmax) bf16 mantissa pairs, at absmax exponents from the
    smallest of the table path (2^-60) to the largest bf16 binade."""
    for e in (-60, -59, -20, -1, 0, 1, 37, 100, 127):
        _write_and_compare(cuda_device, fmt, _ratio_rows(e))
    # below 2^-60 (subnormal scales, clamped codes) the kernel divides
    _write_and_compare(cuda_device, fmt, _ratio_rows(-61))
    _write_and_compare(cuda_device, fmt, _ratio_rows(-126)[::7])


@pytest.mark.parametrize("fmt", ["int8_g64", "int4_g32"])
def test_every_group_quotient_rounds_like_the_oracle(cuda_device, fmt):
    """Grouped formats: every (x, group absmax) bf16 mantissa pair, with the group
    absmax in binary16's subnormal range, across its normal range, at the 65504 clamp
    boundary and beyond it, and at the extremes of bf16."""
    gs = I.GROUPED[fmt]
    for e in (-126, -40, -20, -14, -9, -8, -1, 0, 5, 15, 18, 19, 22, 23, 30, 127):
        _write_and_compare(cuda_device, fmt, _ratio_rows(e, gs))


@pytest.mark.parametrize("scale", [1.0, 0.0625, 2.0 ** -20, 0.05, 0.0112, 3.0, 448.0 / 3])
def test_every_bf16_value_fp8(cuda_device, scale):
    """Every finite bf16 bit pattern through the fp8 write, power-of-two and other scales."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16)
    vals = vals[torch.isfinite(vals.float())]
    pad = (-vals.numel()) % 256
    x = torch.cat([vals, torch.zeros(pad, dtype=torch.bfloat16)]).reshape(-1, 256)
    _write_and_compare(cuda_device, "fp8_e4m3", x, fp8_scale=scale)
