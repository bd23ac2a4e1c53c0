"""The exact top-k + index expansion on the GPU (qsa_topk_expand), through the
C ABI, against the oracle: bit-identical selected slots and cu_seqlens (index
work: no tolerance), at the pages' 8K and 256K context sizes and compress
ratios 4 / 8 / 16, with planted ties, -0.0, -inf and NaN scores, the expansion's
edge lengths, and a page table of 64-token pages; then a captured CUDA graph
replayed with context lengths and scores regenerated on the device (the pages'
"changing-replay index equality"), and the top-k feeding the decode in one graph.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_paged_qsa_gb300 as qsa
from sparse_attention_paged_qsa_gb300 import binding as B
from sparse_attention_paged_qsa_gb300 import inputs as I
from tests.helpers import compare, run_oracle

pytestmark = pytest.mark.gpu

PAGE = 64


def _run(scores, lens, topk, ratio, cap, pt=None, err=None, stream=None):
    dev = scores.device
    bs = lens.numel()
    sel = torch.full((bs * (topk + ratio - 1),), -7, dtype=torch.int32, device=dev)
    cu = torch.full((bs + 1,), -7, dtype=torch.int32, device=dev)
    qsa.qsa_topk_expand(scores, lens, sel, cu, topk, ratio, cap, page_table=pt,
                        page_size=PAGE if pt is not None else 0, error_word=err, stream=stream)
    return sel, cu


def _check(sel, cu, scores, lens, topk, ratio, cap, pt=None, fresh=True):
    want_sel, want_cu = oracle.topk_expand(scores.cpu().numpy(), lens.cpu().numpy(), topk, ratio,
                                           page_table=None if pt is None else pt.cpu().numpy(),
                                           page_size=PAGE, capacity=cap)
    got_cu = cu.cpu().numpy()
    assert got_cu.tolist() == want_cu.tolist()
    got = sel.cpu().numpy()
    assert np.array_equal(got[:got_cu[-1]], want_sel)
    if fresh:  # a buffer filled with -7 before the call: nothing written past the packed rows
        assert (got[got_cu[-1]:] == -7).all()


@pytest.mark.parametrize("cap, bs, ratio, paged", [
    (8192, 16, 4, False), (8192, 16, 8, True), (8192, 16, 16, False),
    (262144, 8, 4, True), (262144, 4, 8, False), (262144, 4, 16, True),
    (4096, 128, 1, False),
])
def test_topk_expand_bit_exact(cuda_device, cap, bs, ratio, paged):
    topk = I.topk_budget(ratio) if ratio > 1 else 1024
    seed = cap // 1024 + bs + ratio
    scores = I.block_scores(bs, cap // ratio, seed, cuda_device)
    lens = I.context_lengths(bs, cap, ratio, topk, seed).to(cuda_device)
    pt = I.page_table(bs, cap, PAGE, seed, cuda_device) if paged else None
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    sel, cu = _run(scores, lens, topk, ratio, cap, pt, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _check(sel, cu, scores, lens, topk, ratio, cap, pt)


def test_topk_expand_saturated_bs128_at_256k(cuda_device):
    cap, ratio, topk, bs = I.TOPK_CAPACITY, I.TOPK_RATIO, I.TOPK_BUDGET, 128
    scores = I.block_scores(bs, cap // ratio, 77, cuda_device)
    lens = torch.full((bs,), cap, dtype=torch.int32, device=cuda_device)
    lens[1::2] = cap - 1                      # rows with the longest tail (3): width 2051
    sel, cu = _run(scores, lens, topk, ratio, cap)
    torch.cuda.synchronize()
    _check(sel, cu, scores, lens, topk, ratio, cap)
    widths = (cu[1:] - cu[:-1]).cpu()
    assert widths.max().item() == oracle.row_width(topk, ratio) == 2051


def test_all_equal_and_all_nan_rows(cuda_device):
    cap, ratio, topk, bs = 65536, 4, 2048, 3
    scores = torch.empty(bs, cap // ratio, device=cuda_device)
    scores[0] = 1.0                  # one tie group: the lowest-indexed blocks are kept
    scores[1] = float("nan")
    scores[2] = -float("inf")
    scores[2, -5:] = float("nan")
    lens = torch.full((bs,), cap, dtype=torch.int32, device=cuda_device)
    sel, cu = _run(scores, lens, topk, ratio, cap)
    torch.cuda.synchronize()
    _check(sel, cu, scores, lens, topk, ratio, cap)
    assert sel[:topk].cpu().tolist() == list(range(topk))


def test_error_flags_clamp_and_do_not_fault(cuda_device):
    cap, ratio, topk, bs = 8192, 4, 2048, 3
    scores = I.block_scores(bs, cap // ratio, 5, cuda_device)
    lens = torch.tensor([cap + 100, -5, 4000], dtype=torch.int32, device=cuda_device)
    pt = I.page_table(bs, cap, PAGE, 5, cuda_device)
    pt[2, 0] = -1                     # slot outside [0, 2^31)
    pt[2, 1] = 1 << 30                # page * 64 overflows int32
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    sel, cu = _run(scores, lens, topk, ratio, cap, pt, err)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & B.DEVERR_CTX_LEN and flags & B.DEVERR_SLOT_RANGE
    # lengths clamped into [0, capacity]; bad page entries give -1 slots
    clamped = torch.tensor([cap, 0, 4000], dtype=torch.int32)
    pt_h = pt.cpu().numpy().astype(np.int64)
    want_sel, want_cu = oracle.topk_expand(scores.cpu().numpy(), clamped.numpy(), topk, ratio,
                                           page_table=np.maximum(pt_h, 0), page_size=PAGE,
                                           capacity=cap)
    got = sel.cpu().numpy()[:want_cu[-1]]
    assert cu.cpu().tolist() == want_cu.tolist()
    bad_pos = (got == -1)
    assert bad_pos.any()
    assert np.array_equal(got[~bad_pos], want_sel[~bad_pos])


def test_sorted_rows_bound_the_first_pass(cuda_device):
    """The first pass stops counting keys below the bin of the first 4096 blocks'
    k-th key once it knows it. Rows sorted descending (the first piece holds the
    row's top keys: the bound is the row's own digit), ascending (the lowest
    bound) and with the top keys only at the end, at 256K contexts through the
    short path (ratio 8), the prefix path (ratio 4) and the no-prefix path (ratio 1)."""
    cap = I.TOPK_CAPACITY
    for ratio, topk in ((8, 2048), (4, 2048), (1, 2048)):
        nbk = cap // ratio
        base = I.block_scores(1, nbk, 40 + ratio, cuda_device, specials=False)[0]
        srt = torch.sort(base, descending=True).values
        late = base.clone()
        late[-3000:] = 5.0 + torch.arange(3000, device=cuda_device, dtype=torch.float32) * 1e-3
        scores = torch.stack([srt, srt.flip(0), late, base])
        # the last: a length whose block count leaves the last bitmap word partly
        # past the row at ratios 4 and 8
        lens = torch.tensor([cap, cap - 3, cap, cap - 8 * 101 - 5], dtype=torch.int32, device=cuda_device)
        sel, cu = _run(scores, lens, topk, ratio, cap)
        torch.cuda.synchronize()
        _check(sel, cu, scores, lens, topk, ratio, cap)


def test_every_cluster_size(cuda_device):
    """Small batches with rows of at least 65,536 blocks take a cluster of CTAs per
    row (8, 4 or 2 by batch size, 1 from 77 rows on a 152-SM GB300): each counts
    and gathers its own part of the row, the leader selects. Rows of full, ragged
    and short lengths at 256K contexts, ratio 4, through a page table, at batch
    sizes that give every cluster size."""
    cap, ratio, topk = I.TOPK_CAPACITY, 4, 2048
    for bs in (1, 20, 40, 77):
        scores = I.block_scores(bs, cap // ratio, 60 + bs, cuda_device)
        lens = torch.full((bs,), cap, dtype=torch.int32)
        lens[1::3] = cap - 8 * 101 - 5        # a part boundary inside the row's last word
        lens[2::3] = 3 * 4096 + 17            # 3,076 blocks: parts of a few words
        lens = lens.to(cuda_device)
        pt = I.page_table(bs, cap, PAGE, 60 + bs, cuda_device)
        err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        sel, cu = _run(scores, lens, topk, ratio, cap, pt, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _check(sel, cu, scores, lens, topk, ratio, cap, pt)


def test_changing_replay_index_equality_in_a_graph(cuda_device):
    """One captured graph: regenerate context lengths and scores on the device from
    the replay counter, then top-k + expansion; 60 replays, every fifth checked
    against the oracle bit for bit."""
    cap, ratio, topk, bs = 65536, 8, 2048, 12
    dev = cuda_device
    scores = torch.empty(bs, cap // ratio, device=dev)
    lens = torch.empty(bs, dtype=torch.int32, device=dev)
    pt = I.page_table(bs, cap, PAGE, 9, dev)
    replay = torch.zeros((), dtype=torch.int64, device=dev)
    sel = torch.empty(bs * (topk + ratio - 1), dtype=torch.int32, device=dev)
    cu = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())

    def body():
        I.replay_context_lengths(11, replay, cap, lens)
        I.replay_block_scores(11, replay, scores)
        qsa.qsa_topk_expand(scores, lens, sel, cu, topk, ratio, cap, page_table=pt,
                            page_size=PAGE, error_word=err, stream=s)
        replay.add_(1)

    with torch.cuda.stream(s):
        body()                       # warm-up outside the capture
    torch.cuda.synchronize()
    replay.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body()
    seen = set()
    for rep in range(60):
        g.replay()
        if rep % 5 == 0:
            torch.cuda.synchronize()
            _check(sel, cu, scores, lens, topk, ratio, cap, pt, fresh=False)
            seen.add(tuple(lens.cpu().tolist()))
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and len(seen) == 12   # the lengths did change every time


def test_cluster_rows_in_a_replayed_graph(cuda_device):
    """The cluster kernel (two 65,536-block rows, 8 CTAs each) captured in a graph:
    lengths and scores regenerated on the device before every replay, every
    replay bit-identical to the oracle."""
    cap, ratio, topk, bs = I.TOPK_CAPACITY, 4, 2048, 2
    dev = cuda_device
    scores = torch.empty(bs, cap // ratio, device=dev)
    lens = torch.empty(bs, dtype=torch.int32, device=dev)
    pt = I.page_table(bs, cap, PAGE, 13, dev)
    replay = torch.zeros((), dtype=torch.int64, device=dev)
    sel = torch.empty(bs * (topk + ratio - 1), dtype=torch.int32, device=dev)
    cu = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())

    def body():
        I.replay_context_lengths(17, replay, cap, lens)
        lens.copy_(cap - torch.remainder(lens, 4096))  # long rows (the cluster path), varying
        I.replay_block_scores(17, replay, scores)
        qsa.qsa_topk_expand(scores, lens, sel, cu, topk, ratio, cap, page_table=pt,
                            page_size=PAGE, error_word=err, stream=s)
        replay.add_(1)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body()
    seen = set()
    for rep in range(8):
        g.replay()
        torch.cuda.synchronize()
        _check(sel, cu, scores, lens, topk, ratio, cap, pt, fresh=False)
        seen.add(tuple(lens.cpu().tolist()))
    assert int(err.item()) == 0 and len(seen) == 8


def test_topk_feeds_the_decode_in_one_graph(cuda_device):
    """Scores -> top-k + expansion (through a page table) -> qsa_decode, one captured
    graph; replays with new scores and lengths; the decode output matches the oracle
    decode of the oracle's own selection."""
    dev = cuda_device
    cap, ratio, topk, bs, hq = 16384, 4, 2048, 6, 24
    npages = bs * (cap // PAGE)
    kc, vc, _, _ = I.make_pools(npages * PAGE, 2, "bf16", seed=21, device=dev)
    q = I.make_query(bs, hq, 21, dev)
    pt = I.page_table(bs, cap, PAGE, 21, dev)
    scores = torch.empty(bs, cap // ratio, device=dev)
    lens = torch.empty(bs, dtype=torch.int32, device=dev)
    replay = torch.zeros((), dtype=torch.int64, device=dev)
    width = topk + ratio - 1
    sel = torch.empty(bs * width, dtype=torch.int32, device=dev)
    cu = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    out = torch.empty(bs, hq, 256, dtype=torch.bfloat16, device=dev)
    scratch = qsa.alloc_scratch(bs, hq, width, dev)
    meta = qsa.KVQuantMeta("bf16", width, None, None, I.SOFTMAX_SCALE)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())

    def body():
        I.replay_context_lengths(5, replay, cap, lens)
        I.replay_block_scores(5, replay, scores)
        qsa.qsa_topk_expand(scores, lens, sel, cu, topk, ratio, cap, page_table=pt,
                            page_size=PAGE, stream=s)
        qsa.qsa_decode(q, kc, vc, meta, sel, cu, out, scratch, s)
        replay.add_(1)

    with torch.cuda.stream(s):
        body()
    torch.cuda.synchronize()
    replay.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body()
    for rep in range(8):
        g.replay()
        if rep % 3 == 0:
            torch.cuda.synchronize()
            _check(sel, cu, scores, lens, topk, ratio, cap, pt, fresh=False)
            n = int(cu[-1].item())
            host = I.host_subset(I.Workload(q, kc, vc, sel[:n].clone(), cu.clone(), "bf16",
                                            capacity=width), list(range(bs)))
            compare(out, run_oracle(host), host.lengths().numpy())
    assert qsa.qsa_scratch_error(scratch) == 0


def test_long_rows_through_every_path(cuda_device):
    """256K contexts (65,536 blocks at ratio 4, 262,144 at ratio 1), longer than the
    kernel keeps as keys in shared memory. At ratio 4 the first pass also keeps the
    keys' top 16 bits: N(0,1) scores leave few enough blocks at or above the k-th
    key's top 11-bit digit to gather those from the prefixes; scores in [1, 1.25)
    with ties (one 11-bit digit) gather from the k-th key's 16-bit prefix instead;
    20,000 scores within 2^-12 of 2 (one 16-bit prefix, the top of the row) take
    the gathered-bin path; scores all within 2^-12 of 1 (every block in one 11-bit
    bin) stream every pass. At ratio 1 (no prefixes) N(0,1) scores take the
    gathered bin."""
    cap = I.TOPK_CAPACITY
    g = torch.Generator(device=cuda_device).manual_seed(3)
    for ratio, topk, kind in ((4, 2048, "normal"), (4, 2048, "crowded"), (4, 2048, "top_cluster"),
                              (4, 2048, "one_bin"), (1, 2048, "normal")):
        bs = 2
        nbk = cap // ratio
        if kind == "crowded":
            scores = 1.0 + 0.25 * torch.rand(bs, nbk, generator=g, device=cuda_device)
            scores[:, ::1000] = 1.125     # and ties inside the crowded bin
        elif kind == "top_cluster":
            scores = torch.randn(bs, nbk, generator=g, device=cuda_device).clamp(-4.0, 1.0)
            idx = torch.randperm(nbk, generator=g, device=cuda_device)[:20000]
            scores[:, idx] = 2.0 + 2.0 ** -12 * torch.rand(bs, 20000, generator=g, device=cuda_device)
        elif kind == "one_bin":
            scores = 1.0 + 2.0 ** -12 * torch.rand(bs, nbk, generator=g, device=cuda_device)
        else:
            scores = I.block_scores(bs, nbk, 31 + ratio, cuda_device)
        lens = torch.tensor([cap, cap - 2], dtype=torch.int32, device=cuda_device)
        sel, cu = _run(scores, lens, topk, ratio, cap)
        torch.cuda.synchronize()
        _check(sel, cu, scores, lens, topk, ratio, cap)
