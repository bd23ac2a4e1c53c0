"""Oracle for the step that produces the decode's selected slots: exact top-k
over compressed-block scores, then index expansion to token slots.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the tests, ``smoke()``
and bench.py's CPU-baseline leg may use it; the product package never imports
it, and it imports nothing from the product package. Plain numpy, index work
only: integers and comparisons of the given float32 scores, no arithmetic on
them.

What the pages fix (1Cat-vLLM PR #523, "Follow-up: device-planned MQA and QSA
quality attribution": "exact top-k + index expansion, fixed 256K capacity", with
compress ratios 4 / 8 / 16; sglang PR #37798, "Decode routing": the index-row
width is token_topk + compress_ratio - 1 = 2048 + 4 - 1 = 2051, and the paged
pool has 64-token pages). What they leave open, and the reading taken here:

* Scores: one float32 per compressed block, given by the caller (the pages give
  no formula for the scoring). Block i of a sequence covers its tokens
  [i r, (i + 1) r), r = the compress ratio; a context of T tokens has floor(T / r)
  complete blocks, and its last T mod r tokens are not yet in a block.
* Top-k: k = token_topk / r blocks are kept: every block when there are at most
  k, otherwise the k ranked first, where a higher score ranks first, equal scores
  rank by lower block index, NaN ranks below every number (-inf included), and
  -0.0 equals +0.0.
* Expansion: the tokens of the kept blocks in ascending position, then the tail
  tokens (those not yet in a block), so a row holds at most token_topk + r - 1
  ids, the pages' width.
* Slots: with a page table, the token at logical position p of sequence b is
  slot page_table[b][p // page] * page + p % page; without one, the id is p.
* Rows are packed one after another; cu_seqlens[b] is where row b starts
  (cu_seqlens[0] = 0), the layout the decode takes.
"""
from __future__ import annotations

import numpy as np


class TopkRefused(ValueError):
    """The input breaks the contract (bad lengths, sizes or page table)."""


def topk_blocks(scores_row, nb: int, kb: int) -> np.ndarray:
    """Ascending indices of the blocks kept among the first nb scores of a row."""
    if nb <= kb:
        return np.arange(nb, dtype=np.int64)
    s = np.asarray(scores_row[:nb], dtype=np.float32).astype(np.float64) + 0.0  # -0.0 -> +0.0
    nan = np.isnan(s)
    filled = np.where(nan, 0.0, s)
    # rank: non-NaN before NaN, then score descending, then block index ascending
    order = np.lexsort((np.arange(nb), -filled, nan))
    return np.sort(order[:kb])


def expand(blocks: np.ndarray, T: int, ratio: int) -> np.ndarray:
    """Logical token positions of a row: each kept block's r tokens, then the tail."""
    nb = T // ratio
    pos = (np.asarray(blocks, np.int64)[:, None] * ratio + np.arange(ratio)[None, :]).reshape(-1)
    return np.concatenate([pos, np.arange(nb * ratio, T, dtype=np.int64)])


def topk_expand(scores, ctx_lens, token_topk: int, ratio: int, page_table=None,
                page_size: int = 64, capacity: int = 262144):
    """Selected slots of every sequence, packed: returns (sel int32 [n], cu int32 [bs + 1]).

    scores:     float32 [bs, >= capacity // ratio], one score per compressed block
    ctx_lens:   int [bs], context length T_b in tokens, 0 <= T_b <= capacity
    page_table: optional int [bs, >= ceil(capacity / page_size)] physical page ids
    """
    if ratio < 1 or token_topk < ratio or token_topk % ratio:
        raise TopkRefused("token_topk must be a positive multiple of the compress ratio")
    scores = np.asarray(scores, dtype=np.float32)
    lens = np.asarray(ctx_lens, dtype=np.int64)
    bs = lens.shape[0]
    kb = token_topk // ratio
    parts, cu = [], [0]
    for b in range(bs):
        T = int(lens[b])
        if T < 0 or T > capacity or T // ratio > scores.shape[1]:
            raise TopkRefused(f"context length {T} of sequence {b} outside the contract")
        pos = expand(topk_blocks(scores[b], T // ratio, kb), T, ratio)
        if page_table is not None:
            pt = np.asarray(page_table[b], dtype=np.int64)
            if pos.size and (pos[-1] // page_size >= pt.shape[0]):
                raise TopkRefused("page table too short")
            pos = pt[pos // page_size] * page_size + pos % page_size
        parts.append(pos)
        cu.append(cu[-1] + pos.size)
    sel = np.concatenate(parts) if parts else np.zeros(0, np.int64)
    return sel.astype(np.int32), np.asarray(cu, dtype=np.int32)


def row_width(token_topk: int, ratio: int) -> int:
    """Longest row the expansion can produce: k r block tokens and r - 1 tail tokens."""
    return token_topk + ratio - 1
