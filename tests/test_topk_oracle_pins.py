"""Pins for the top-k + index-expansion oracle (oracle/topk.py).

Each test checks the oracle against something other than itself: a worked
example derived by hand from the definition, brute force over every subset on
tiny inputs (the kept set defined as the one no left-out block outranks, not by
sorting), torch.topk on distinct scores, the pages' row width, and properties
at the pages' 256K capacity. A plausible slip -- ties broken by the higher
index, NaN ranked above -inf, -0.0 below +0.0, the tail dropped or shifted, a
block expanded to the wrong tokens, a wrong page mapping -- fails one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAN, INF = float("nan"), float("inf")


def _ranks_before(a, i, b, j):
    """True when block i (score a) ranks before block j (score b): higher first,
    NaN below every number, -0.0 == +0.0, ties by lower index."""
    if math.isnan(a) != math.isnan(b):
        return math.isnan(b)
    if math.isnan(a) or a == b:
        return i < j
    return a > b


def test_worked_example_by_hand():
    # r = 4, token_topk = 8 -> 2 blocks kept; rows padded with junk past T // r
    scores = np.array([
        [1.0, 3.0, 1.0, 1.0, NAN, -INF, 9.0],   # T=27: 6 blocks, tail 24..26
        [NAN, NAN, 7.0, 7.0, 7.0, 7.0, 7.0],     # T=9: 2 blocks <= 2 -> all, tail 8
        [-0.0, 0.0, 0.0, -1.0, 9.0, 9.0, 9.0],   # T=16: 4 blocks, no tail
        [NAN, -INF, NAN, -INF, 5.0, 9.0, 9.0],   # T=20: 5 blocks, no tail
        [9.0] * 7,                                # T=0: empty row
        [9.0] * 7,                                # T=3: no block, tail 0..2
    ], dtype=np.float32)
    lens = [27, 9, 16, 20, 0, 3]
    sel, cu = oracle.topk_expand(scores, lens, token_topk=8, ratio=4, capacity=28)
    rows = [sel[cu[b]:cu[b + 1]].tolist() for b in range(len(lens))]
    # 3.0 (block 1) first; the tie at 1.0 goes to the lowest index (block 0), not 2 or 3
    assert rows[0] == [0, 1, 2, 3, 4, 5, 6, 7, 24, 25, 26]        # width 8 + 4 - 1 = 11
    assert rows[1] == list(range(9))
    # -0.0 equals +0.0, so blocks 0 and 1 (ties by index), not 1 and 2
    assert rows[2] == list(range(8))
    # 5.0 (block 4), then the -inf blocks 1 and 3 outrank the NaN blocks: block 1
    assert rows[3] == [4, 5, 6, 7, 16, 17, 18, 19]
    assert rows[4] == [] and rows[5] == [0, 1, 2]
    assert cu.tolist() == [0, 11, 20, 28, 36, 36, 39]
    # the same through a page table of 4-slot pages
    pt = np.array([[7, 2, 9, 0, 5, 1, 3]] * 6)
    sel_p, cu_p = oracle.topk_expand(scores, lens, 8, 4, page_table=pt, page_size=4, capacity=28)
    assert sel_p[:11].tolist() == [28, 29, 30, 31, 8, 9, 10, 11, 12, 13, 14]
    assert cu_p.tolist() == cu.tolist()


def test_row_width_is_the_pages():
    for line in open(os.path.join(GOLDEN, "topk_row_width.txt")):
        if line.startswith("#") or not line.strip():
            continue
        topk, ratio, width = map(int, line.split())
        assert oracle.row_width(topk, ratio) == width
        # reached when at least topk / ratio blocks exist and the tail is ratio - 1 long
        T = 4 * topk + ratio - 1
        scores = np.random.default_rng(0).standard_normal((1, T // ratio)).astype(np.float32)
        sel, cu = oracle.topk_expand(scores, [T], topk, ratio)
        assert cu[1] - cu[0] == width


@pytest.mark.parametrize("seed", range(40))
def test_kept_set_equals_brute_force_over_subsets(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 8))
    kb = int(rng.integers(1, 5))
    ratio = int(rng.choice([1, 2, 4]))
    pool = np.array([NAN, -INF, -1.0, -0.0, 0.0, 0.5, 1.0, INF], dtype=np.float32)
    s = pool[rng.integers(0, len(pool), nb)]
    T = nb * ratio + int(rng.integers(0, ratio))
    sel, cu = oracle.topk_expand(s[None, :], [T], kb * ratio, ratio, capacity=T)
    got = sorted({int(p) // ratio for p in sel if p < nb * ratio})
    # brute force: the kept set is the size-min(nb, kb) subset that no left-out block outranks
    want = []
    for sub in itertools.combinations(range(nb), min(nb, kb)):
        out = [j for j in range(nb) if j not in sub]
        if all(not _ranks_before(float(s[j]), j, float(s[i]), i) for i in sub for j in out):
            want.append(list(sub))
    assert len(want) == 1, want
    assert got == want[0]


def test_distinct_scores_match_torch_topk():
    rng = np.random.default_rng(1)
    for nb, kb in ((2048, 512), (65536, 512), (700, 699)):
        s = rng.permutation(nb).astype(np.float32) * 0.25 - 100.0   # distinct, exact in fp32
        blocks = oracle.topk_blocks(s, nb, kb)
        ref = torch.topk(torch.from_numpy(s), kb).indices.numpy()
        assert sorted(ref.tolist()) == blocks.tolist()


def test_properties_at_the_256k_capacity():
    rng = np.random.default_rng(2)
    ratio, topk, cap = 4, 2048, 262144
    bs = 3
    scores = rng.standard_normal((bs, cap // ratio)).astype(np.float32)
    scores[0, ::97] = 0.5             # a large tie group
    scores[1, ::13] = -np.inf
    scores[1, ::29] = np.nan
    lens = [cap, cap - 1, 8191]
    sel, cu = oracle.topk_expand(scores, lens, topk, ratio, capacity=cap)
    kb = topk // ratio
    for b, T in enumerate(lens):
        row = sel[cu[b]:cu[b + 1]].astype(np.int64)
        nb = T // ratio
        assert row.size == ratio * min(nb, kb) + T % ratio
        assert (np.diff(row) > 0).all() and row[0] >= 0 and row[-1] < T
        body = row[: ratio * min(nb, kb)].reshape(-1, ratio)
        assert (body == body[:, :1] + np.arange(ratio)).all() and (body[:, 0] % ratio == 0).all()
        assert row[ratio * min(nb, kb):].tolist() == list(range(nb * ratio, T))
        kept = body[:, 0] // ratio
        s = scores[b, :nb].astype(np.float64)
        mask = np.zeros(nb, bool)
        mask[kept] = True
        key = np.where(np.isnan(s), -np.inf, s)
        # no left-out block outranks a kept one
        assert key[mask].min() >= key[~mask].max()
        thr = key[mask].min()
        assert not (np.isnan(s[mask]).any() and (~np.isnan(s[~mask])).any())
        ties_out = np.flatnonzero(~mask & (key == thr) & ~np.isnan(s))
        ties_in = np.flatnonzero(mask & (key == thr) & ~np.isnan(s))
        if ties_out.size and ties_in.size:
            assert ties_in.max() < ties_out.min()


def test_page_table_mapping_and_refusals():
    rng = np.random.default_rng(3)
    T, ratio, topk, page = 1000, 8, 64, 64
    scores = rng.standard_normal((1, T // ratio)).astype(np.float32)
    pages = rng.permutation(1000)[:16]
    plain, _ = oracle.topk_expand(scores, [T], topk, ratio, capacity=1024)
    paged, _ = oracle.topk_expand(scores, [T], topk, ratio, page_table=pages[None, :],
                                  page_size=page, capacity=1024)
    assert paged.tolist() == [int(pages[p // page]) * page + p % page for p in plain.tolist()]
    with pytest.raises(oracle.TopkRefused):
        oracle.topk_expand(scores, [T], 60, ratio)            # not a multiple of the ratio
    with pytest.raises(oracle.TopkRefused):
        oracle.topk_expand(scores, [T + 8], topk, ratio, capacity=1024)   # past the scores
    with pytest.raises(oracle.TopkRefused):
        oracle.topk_expand(scores, [T], topk, ratio, capacity=999)        # past the capacity
