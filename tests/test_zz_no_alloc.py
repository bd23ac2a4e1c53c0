"""qsa_decode_static_scratch: decode without a caller-provided scratch buffer.

This entry point serves callers that cannot allocate device memory when they
call (fixed-budget plugins, allocator-less bindings, loops where an
allocation would synchronise the device): its scratch is a fixed device array
inside libqsa. Here it is called through the C ABI, twice in a row on
different workloads; each result must match qsa_decode (which uses a
caller-allocated scratch buffer) within the parity tolerance, and each is also
checked against the FP64 oracle with the suite's degenerate-output rejections,
so a fault shared by both entry points cannot pass unnoticed.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_paged_qsa_gb300 import binding as B
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import REL_L2_TOL, compare, rel_l2, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


def _call_static(wd, out, max_ctas=0):
    lib = B.load()
    meta = B.KVQuantMeta(wd.fmt, wd.capacity, wd.k_scale, wd.v_scale, wd.softmax_scale,
                         max_ctas).to_c()
    d = [B.describe(t) for t in (wd.q, wd.k_pool, wd.v_pool, wd.sel, wd.cu, out)]
    rc = lib.qsa_decode_static_scratch(
        ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[2]), ctypes.byref(meta),
        ctypes.byref(d[3]), ctypes.byref(d[4]), ctypes.byref(d[5]),
        torch.cuda.current_stream().cuda_stream)
    return rc, lib.qsa_last_error_message().decode()


def _matches(a: torch.Tensor, b: torch.Tensor) -> float:
    x = a.float().cpu().double().numpy()
    y = b.float().cpu().double().numpy()
    assert np.isfinite(x).all()
    err = rel_l2(x, y)
    return float(err.max())


def test_static_scratch_matches_qsa_decode_on_two_calls(cuda_device):
    hosts = (I.tp1_mixed(seed=31, bs=16, num_slots=65536),
             I.tiny_tp2(seed=32, length=2055, fmt="int8"))
    for w in hosts:
        wd = w.to(cuda_device)
        ref, _ = run_cuda(wd)
        out = torch.full_like(wd.q, float("nan"))
        rc, msg = _call_static(wd, out)
        assert rc == B.OK, msg
        torch.cuda.synchronize()
        assert _matches(out, ref) <= REL_L2_TOL
        compare(out, run_oracle(w), w.lengths().numpy())


def test_static_scratch_rejects_sizes_beyond_its_limit(cuda_device):
    w = I.tiny_tp2(seed=33, length=16).to(cuda_device)
    big = I.Workload(torch.zeros(129, 12, 256, dtype=torch.bfloat16, device=cuda_device),
                     w.k_pool, w.v_pool, w.sel,
                     torch.zeros(130, dtype=torch.int32, device=cuda_device), "bf16",
                     capacity=16)
    out = torch.empty_like(big.q)
    rc, msg = _call_static(big, out)
    assert rc == B.ERR_UNSUPPORTED and "batch size" in msg
