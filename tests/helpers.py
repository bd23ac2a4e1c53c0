"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle,
compare per (sequence, head)."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import inputs as I

# Gate from the pages: relative L2 <= 2e-3 per (sequence, head) against an
# independent FP32 reference (sglang PR #36845, "Optimized kernel"); here the
# reference is the FP64 oracle rounded to bf16 like the output.
REL_L2_TOL = 2e-3


def meta_for(w: I.Workload, max_ctas: int = 0, capacity=None) -> qsa.KVQuantMeta:
    tier = {k: w.extra[k] for k in I.TIER_KEYS} if w.fmt == I.TIERED else None
    return qsa.KVQuantMeta(w.fmt, capacity or w.capacity, w.k_scale, w.v_scale, w.softmax_scale,
                           max_ctas, tier)


def run_cuda(wd: I.Workload, max_ctas: int = 0, out=None, scratch=None, stream=None):
    """qsa_decode on a device-resident workload; returns (out, scratch)."""
    if out is None:
        out = torch.full_like(wd.q, float("nan"))
    if scratch is None:
        scratch = qsa.alloc_scratch(wd.bs, wd.num_q_heads, wd.capacity, wd.q.device)
    qsa.qsa_decode(wd.q, wd.k_pool, wd.v_pool, meta_for(wd, max_ctas), wd.sel, wd.cu, out,
                   scratch, stream)
    return out, scratch


def run_oracle(w: I.Workload, rows=None) -> np.ndarray:
    """FP64 oracle output [n, Hq, 256] on a host workload."""
    if w.fmt == I.TIERED:
        t = w.extra
        return oracle.decode_tiered(w.q, w.k_pool, w.v_pool, w.sel, w.cu, w.softmax_scale,
                                    w.k_scale, w.v_scale, t["k_ring"], t["v_ring"],
                                    t["k_ring_scale"], t["v_ring_scale"], t["owner"], rows=rows)
    return oracle.decode(w.q, w.k_pool, w.v_pool, w.fmt, w.sel, w.cu, w.softmax_scale,
                         w.k_scale, w.v_scale, rows=rows)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per-(sequence, head) relative L2 over the head dimension; rows whose
    reference is zero must match exactly (reported as 0 or inf)."""
    num = np.sqrt(((got - ref) ** 2).sum(-1))
    den = np.sqrt((ref ** 2).sum(-1))
    out = np.where(den > 0, num / np.where(den > 0, den, 1), np.where(num > 0, np.inf, 0.0))
    return out


def compare(got_bf16: torch.Tensor, ref64: np.ndarray, lengths, rows=None, tol=REL_L2_TOL):
    """Check a CUDA bf16 output against the oracle; returns (max rel-L2 vs
    bf16(oracle), max rel-L2 vs unrounded oracle)."""
    got = got_bf16.float().cpu().double().numpy()
    if rows is not None:
        got = got[np.asarray(rows)]
        lengths = np.asarray(lengths)[np.asarray(rows)]
    assert np.isfinite(got).all(), "non-finite output"
    lengths = np.asarray(lengths)
    # degenerate-output rejection (the pages' failure mode was all-token-0 output)
    live = lengths > 0
    if live.any():
        assert (np.abs(got[live]).sum(-1) > 0).all(), "all-zero output row for a live sequence"
    if live.sum() > 1:
        flat = got[live].reshape(live.sum(), -1)
        assert not (flat == flat[:1]).all(), "identical outputs across sequences"
    assert (got[~live] == 0).all(), "empty selection must give zeros"
    ref_b = oracle.round_bf16(ref64)
    e_b = rel_l2(got, ref_b)
    e_u = rel_l2(got, ref64)
    finite_u = e_u[np.isfinite(e_u)]
    REPORT.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], float(e_b.max()),
                   float(finite_u.max()) if finite_u.size else 0.0))
    assert e_b.max() <= tol, f"rel-L2 {e_b.max():.3e} > {tol} (worst at {np.unravel_index(e_b.argmax(), e_b.shape)})"
    return float(e_b.max()), float(e_u.max())


# (test, max rel-L2 vs bf16(oracle), max rel-L2 vs the unrounded oracle) of every
# compare() in this session; the terminal summary prints them (tests/conftest.py)
REPORT = []


def counters(scratch: torch.Tensor, bs: int, hq: int, capacity: int) -> torch.Tensor:
    ly = qsa.qsa_decode_scratch_layout(bs, hq, capacity)
    off, n = ly["counters_offset"], ly["counters_count"]
    return scratch[off:off + 4 * n].view(torch.int32).cpu()


gather_subset = I.host_subset
