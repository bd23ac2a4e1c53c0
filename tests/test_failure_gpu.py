"""Bounded pipeline waits on the GPU: a wait that runs out ends the launch with
an error status the host reads, and the context stays usable.

The test build of the decode (libqsa_testhooks.so, compiled with
-DQSA_TEST_HOOKS; the shipped libqsa.so has no hook) exports
qsa_test_set_stall_stage(k): CTA 0's producer warps then leave their k-th stage
incomplete (they never arrive on its mbarrier), so the consumer warps' wait for
it runs out after its limit (2 s of %globaltimer).
Nothing traps, faults or spins without a limit: the consumers record
QSA_DEVERR_TIMEOUT, raise the CTA's abort flag and leave, and the producers'
own bounded waits then end too. After re-zeroing the scratch the next call is
checked against the oracle.
"""
import ctypes
import os
import time

import pytest
import torch

import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import binding as B
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, counters, run_oracle

pytestmark = pytest.mark.gpu

DEVERR_TIMEOUT = 4


def _decode(lib, wd, meta, out, scratch):
    m = meta.to_c()
    d = [B.describe(t) for t in (wd.q, wd.k_pool, wd.v_pool, wd.sel, wd.cu, out)]
    rc = lib.qsa_decode(ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[2]), ctypes.byref(m),
                        ctypes.byref(d[3]), ctypes.byref(d[4]), ctypes.byref(d[5]),
                        scratch.data_ptr(), scratch.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == B.OK, lib.qsa_last_error_message().decode()


def test_stalled_stage_times_out_and_context_recovers(cuda_device):
    lib = B.open_library(os.path.join(os.path.dirname(B.LIB_PATH), "libqsa_testhooks.so"))
    lib.qsa_test_set_stall_stage.argtypes = [ctypes.c_int]
    w = I.tp1_mixed(seed=23, bs=16, num_slots=65536)
    wd = w.to(cuda_device)
    # CTA 0 streams several stages, so its stage 1 exists
    n_tokens = int(w.lengths().sum()) * 2
    grid = qsa.qsa_decode_grid(w.bs, w.num_q_heads, w.capacity)
    assert n_tokens // grid >= 2 * 64
    meta = qsa.KVQuantMeta("bf16", w.capacity, None, None, w.softmax_scale)
    out = torch.zeros_like(wd.q)
    scratch = qsa.alloc_scratch(w.bs, w.num_q_heads, w.capacity, cuda_device)

    lib.qsa_test_set_stall_stage(1)
    t0 = time.monotonic()
    try:
        _decode(lib, wd, meta, out, scratch)
        torch.cuda.synchronize()
    finally:
        lib.qsa_test_set_stall_stage(-1)
    waited = time.monotonic() - t0
    assert qsa.qsa_scratch_error(scratch, clear=True) & DEVERR_TIMEOUT
    assert 1.0 < waited < 60.0, waited  # the wait ran out at its limit, not before

    # the context is usable: zero the scratch (split counters may be mid-count) and decode again
    qsa.qsa_scratch_init(scratch)
    out.zero_()
    _decode(lib, wd, meta, out, scratch)
    torch.cuda.synchronize()
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    compare(out, run_oracle(w), w.lengths().numpy())


def test_stalled_contributor_of_an_equal_length_split_times_out(cuda_device):
    """bs = 1, L = 2055 (equal lengths, 16 CTAs per KV head, each merging a slice of
    its segment once all 16 partials are stored): CTA 0 never completes its second
    stage and leaves without a partial; the other contributors' bounded wait for
    the sixteenth ticket runs out, and the launch ends with the timeout status."""
    lib = B.open_library(os.path.join(os.path.dirname(B.LIB_PATH), "libqsa_testhooks.so"))
    lib.qsa_test_set_stall_stage.argtypes = [ctypes.c_int]
    w = I.tp1_mixed(seed=24, bs=1, num_slots=65536, lengths=[2055])
    wd = w.to(cuda_device)
    meta = qsa.KVQuantMeta("bf16", w.capacity, None, None, w.softmax_scale)
    out = torch.zeros_like(wd.q)
    scratch = qsa.alloc_scratch(w.bs, w.num_q_heads, w.capacity, cuda_device)

    lib.qsa_test_set_stall_stage(1)
    t0 = time.monotonic()
    try:
        _decode(lib, wd, meta, out, scratch)
        torch.cuda.synchronize()
    finally:
        lib.qsa_test_set_stall_stage(-1)
    waited = time.monotonic() - t0
    assert qsa.qsa_scratch_error(scratch, clear=True) & DEVERR_TIMEOUT
    assert 1.0 < waited < 60.0, waited

    qsa.qsa_scratch_init(scratch)
    out.zero_()
    _decode(lib, wd, meta, out, scratch)
    torch.cuda.synchronize()
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    compare(out, run_oracle(w), w.lengths().numpy())
