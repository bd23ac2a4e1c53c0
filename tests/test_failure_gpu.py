"""Bounded pipeline waits on the GPU: a wait that runs out ends the launch with
an error status the host reads, and the context stays usable.

The library's test hook QSA_TEST_STALL_STAGE=k makes CTA 0's producer warps
leave their k-th stage incomplete (they never arrive on its mbarrier), so the
consumer warps' wait for it runs out after its limit (2 s of %globaltimer).
Nothing traps, faults or spins without a limit: the consumers record
QSA_DEVERR_TIMEOUT, raise the CTA's abort flag and leave, and the producers'
own bounded waits then end too. After re-zeroing the scratch the next call is
checked against the oracle.
"""
import time

import pytest
import torch

import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, counters, run_oracle

pytestmark = pytest.mark.gpu

DEVERR_TIMEOUT = 4


def test_stalled_stage_times_out_and_context_recovers(cuda_device, monkeypatch):
    w = I.tp1_mixed(seed=23, bs=16, num_slots=65536)
    wd = w.to(cuda_device)
    # CTA 0 streams several stages, so its stage 1 exists
    n_tokens = int(w.lengths().sum()) * 2
    grid = qsa.qsa_decode_grid(w.bs, w.num_q_heads, w.capacity)
    assert n_tokens // grid >= 2 * 64
    meta = qsa.KVQuantMeta("bf16", w.capacity, None, None, w.softmax_scale)
    out = torch.zeros_like(wd.q)
    scratch = qsa.alloc_scratch(w.bs, w.num_q_heads, w.capacity, cuda_device)

    monkeypatch.setenv("QSA_TEST_STALL_STAGE", "1")
    t0 = time.monotonic()
    qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta, wd.sel, wd.cu, out, scratch)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    monkeypatch.delenv("QSA_TEST_STALL_STAGE")
    assert qsa.qsa_scratch_error(scratch, clear=True) & DEVERR_TIMEOUT
    assert 1.0 < waited < 60.0, waited  # the wait ran out at its limit, not before

    # the context is usable: zero the scratch (split counters may be mid-count) and decode again
    qsa.qsa_scratch_init(scratch)
    out.zero_()
    qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta, wd.sel, wd.cu, out, scratch)
    torch.cuda.synchronize()
    assert qsa.qsa_scratch_error(scratch) == 0
    assert (counters(scratch, w.bs, w.num_q_heads, w.capacity) == 0).all()
    compare(out, run_oracle(w), w.lengths().numpy())
