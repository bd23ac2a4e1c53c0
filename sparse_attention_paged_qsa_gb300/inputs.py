"""Seeded synthetic inputs for packed QSA decode.

This module is shared by the GPU tests, the benchmark and the oracle tests.
It holds input generation only -- random pools, queries, selected-slot lists
and cu_seqlens, and the KV-write-side quantisers that turn N(0,1) draws into
the fp8 / int8 / int4 pool formats. It contains none of the decode
arithmetic (no dequantisation, no scores, no softmax); neither the CUDA
path nor the oracle is imported here.

Workload shapes follow the pages: one BF16 query token per sequence with
24 query / 2 KV heads (TP1) or 12 / 1 (TP2), head dim 256, a paged pool with
64-token pages and per-sequence selections of up to 2055 slots (sglang PR
#36845, "Changes"; sglang PR #37798, "Decode routing": page 64, top-k
2048 + 4 - 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

HEAD_DIM = 256
GQA_GROUP = 12          # query heads per KV head (12:1 GQA)
PAGE = 64               # slots per page
MAX_CAPACITY = 2055     # largest selected-KV length of the contract
SOFTMAX_SCALE = 1.0 / 16.0

FORMATS = ("bf16", "fp8_e4m3", "int8", "int4", "int8_g64", "int4_g32")
TIERED = "int8ring_int4"   # int4_g32 pool of every slot + int8_g64 ring with an owner table
RING_SLOTS = 8192          # the pages' default ring size
TIER_KEYS = ("k_ring", "v_ring", "k_ring_scale", "v_ring_scale", "owner")
GROUPED = {"int8_g64": 64, "int4_g32": 32}   # channels per binary16 scale
NIBBLE_FORMATS = ("int4", "int4_g32")        # two 4-bit codes per byte
FP8_E4M3_MAX = 448.0    # largest finite e4m3fn value; the fp8 write saturates here
FP16_MAX = 65504.0      # the grouped formats' scale clamp (largest finite binary16)


@dataclass
class Workload:
    """One decode call's inputs (all tensors on one device)."""

    q: torch.Tensor                  # [bs, Hq, 256] bf16
    k_pool: torch.Tensor             # [slots, Hkv, 256] bf16/uint8/int8 or [slots, Hkv, 128] uint8
    v_pool: torch.Tensor
    sel: torch.Tensor                # int32 [n_sel], packed by cu
    cu: torch.Tensor                 # int32 [bs+1]
    fmt: str = "bf16"
    k_scale: Optional[torch.Tensor] = None   # fp8: [1]; int8/int4: [slots, Hkv] float32;
                                             # grouped: [slots, Hkv, 256 / group] float16
    v_scale: Optional[torch.Tensor] = None
    softmax_scale: float = SOFTMAX_SCALE
    capacity: int = MAX_CAPACITY
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def bs(self) -> int:
        return self.q.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_pool.shape[1]

    @property
    def num_slots(self) -> int:
        return self.k_pool.shape[0]

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        extra = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.extra.items()}
        return Workload(mv(self.q), mv(self.k_pool), mv(self.v_pool), mv(self.sel), mv(self.cu),
                        self.fmt, mv(self.k_scale), mv(self.v_scale), self.softmax_scale,
                        self.capacity, self.name, extra)

    def lengths(self) -> torch.Tensor:
        return (self.cu[1:] - self.cu[:-1]).cpu()


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


# ---------------------------------------------------------------- pool values

def normal_values(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """float32 N(0, std^2) draws from torch's seeded generator on `device`."""
    return torch.randn(shape, generator=_gen(seed, device), device=device,
                       dtype=torch.float32) * std


def quantize_pool(x: torch.Tensor, fmt: str):
    """KV-write-side quantiser (input generation): float32 [slots, Hkv, D] -> (codes, scale).

    fp8 : one fp32 scale per pool = absmax / 448; codes = e4m3fn(clamp(x / s, +-448))
          (the clamp mirrors the fp8 write path's saturation before the cast,
          sglang PR #37798 part 1, "mem_cache/memory_pool.py").
    int8: fp32 scale per (slot, KV head) = absmax(row) / 127; codes = clamp(rint(x/s), -127, 127).
    int4: fp32 scale per (slot, KV head) = absmax(row) / 7; codes = clamp(rint(x/s), -8, 7),
          two's-complement nibbles, two per byte, element 2i in the low nibble.
    int8_g64 / int4_g32 (sglang PR #37798, "Modifications", the int8 and int4 KV
          pool modules): per 64 / 32-channel group a binary16 scale
          s16 = fp16(min(absmax / q, 65504)), q = 127 / 7; codes = clamp(rint(x / s16), -q, q);
          int4_g32 stores offset-binary nibbles code + 8, element 2i in the low nibble.
    rint is round-half-to-even (torch.round). A zero row gets scale 0 and zero codes.
    """
    if fmt == "bf16":
        return x.to(torch.bfloat16), None
    if fmt == "fp8_e4m3":
        amax = x.abs().max().to(torch.float32)
        s = (amax / FP8_E4M3_MAX).reshape(1)
        y = torch.where(s > 0, x / s, torch.zeros_like(x)).clamp(-FP8_E4M3_MAX, FP8_E4M3_MAX)
        return y.to(torch.float8_e4m3fn).view(torch.uint8), s.to(torch.float32)
    if fmt in ("int8", "int4"):
        qmax = 127.0 if fmt == "int8" else 7.0
        qmin = -127.0 if fmt == "int8" else -8.0
        amax = x.abs().amax(dim=-1)
        s = (amax / qmax).to(torch.float32)
        safe = torch.where(s > 0, s, torch.ones_like(s)).unsqueeze(-1)
        qv = torch.where(s.unsqueeze(-1) > 0, torch.round(x / safe), torch.zeros_like(x))
        qv = qv.clamp(qmin, qmax).to(torch.int8)
        if fmt == "int8":
            return qv, s
        lo = (qv[..., 0::2].to(torch.int16) & 0xF)
        hi = (qv[..., 1::2].to(torch.int16) & 0xF)
        return (lo | (hi << 4)).to(torch.uint8), s
    if fmt in GROUPED:
        gs = GROUPED[fmt]
        qmax = 127.0 if fmt == "int8_g64" else 7.0
        xg = x.reshape(*x.shape[:-1], x.shape[-1] // gs, gs)
        amax = xg.abs().amax(dim=-1)
        s16 = (amax / qmax).to(torch.float32).clamp(max=FP16_MAX).to(torch.float16)
        s32 = s16.to(torch.float32).unsqueeze(-1)
        safe = torch.where(s32 > 0, s32, torch.ones_like(s32))
        qv = torch.where(s32 > 0, torch.round(xg / safe), torch.zeros_like(xg))
        qv = qv.clamp(-qmax, qmax).to(torch.int8).reshape(x.shape)
        if fmt == "int8_g64":
            return qv, s16
        u = qv.to(torch.int16) + 8
        return (u[..., 0::2] | (u[..., 1::2] << 4)).to(torch.uint8), s16
    raise ValueError(f"unknown pool format {fmt!r}")


def make_pools(num_slots: int, num_kv_heads: int, fmt: str, seed: int, device="cpu"):
    """K and V pools [slots, Hkv, 256] from N(0,1) draws, in pool format `fmt`.

    Returns (k_codes, v_codes, k_scale, v_scale)."""
    shape = (num_slots, num_kv_heads, HEAD_DIM)
    kx = normal_values(shape, seed * 1000 + 1, device)
    kc, ks = quantize_pool(kx, fmt)
    del kx
    vx = normal_values(shape, seed * 1000 + 2, device)
    vc, vs = quantize_pool(vx, fmt)
    del vx
    return kc, vc, ks, vs


def make_tiered_pools(num_slots: int, num_kv_heads: int, ring_slots: int, seed: int, device="cpu",
                      unowned: float = 0.1):
    """A tiered int8ring_int4 pool as a run of writes leaves it (sglang PR #37798,
    "Modifications", the tiered KV pool module): every slot holds its int4_g32 row;
    slots were written in a seeded random order, so ring position p holds the int8_g64
    row of the last slot written with slot & (R - 1) == p, and owner[p] is that slot.
    A share `unowned` of ring positions was never written (owner -1, ring rows zero).

    Returns (k_pool, v_pool, k_scale, v_scale, tier) with tier a dict of TIER_KEYS."""
    if ring_slots <= 0 or ring_slots & (ring_slots - 1):
        raise ValueError("the ring size must be a power of two")
    shape = (num_slots, num_kv_heads, HEAD_DIM)
    g = torch.Generator().manual_seed(seed * 1000 + 7)
    order = torch.randperm(num_slots, generator=g)
    pos = order & (ring_slots - 1)
    last = torch.full((ring_slots,), -1, dtype=torch.int64)
    last.scatter_reduce_(0, pos, torch.arange(num_slots), reduce="amax")   # latest write per position
    owner = torch.where(last >= 0, order[last.clamp(min=0)], torch.full_like(last, -1))
    drop = torch.rand(ring_slots, generator=g) < unowned
    owner = torch.where(drop, torch.full_like(owner, -1), owner).to(torch.int32)
    out = {}
    for name, sub in (("k", 1), ("v", 2)):
        x = normal_values(shape, seed * 1000 + sub, device)
        codes4, s4 = quantize_pool(x, "int4_g32")
        own = owner.to(device).long()
        rows = x.index_select(0, own.clamp(min=0))
        codes8, s8 = quantize_pool(rows, "int8_g64")
        live = (own >= 0).view(-1, 1, 1)
        out[name] = (codes4, s4, torch.where(live, codes8, torch.zeros_like(codes8)),
                     torch.where(live, s8, torch.zeros_like(s8)))
        del x, rows
    tier = {"k_ring": out["k"][2], "v_ring": out["v"][2], "k_ring_scale": out["k"][3],
            "v_ring_scale": out["v"][3], "owner": owner.to(device)}
    return out["k"][0], out["v"][0], out["k"][1], out["v"][1], tier


def make_query(bs: int, num_q_heads: int, seed: int, device="cpu") -> torch.Tensor:
    return normal_values((bs, num_q_heads, HEAD_DIM), seed * 1000 + 3, device).to(torch.bfloat16)


# ---------------------------------------------------------- selected slots

def cu_from_lengths(lengths) -> torch.Tensor:
    lens = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lens.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    return cu.to(torch.int32)


def uniform_indices(n: int, num_slots: int, gen: torch.Generator) -> torch.Tensor:
    """n slot ids drawn uniformly with replacement (duplicates kept, order as drawn)."""
    return torch.randint(0, num_slots, (n,), generator=gen, dtype=torch.int64).to(torch.int32)


def runs_and_uniform_indices(length: int, num_slots: int, gen: torch.Generator) -> torch.Tensor:
    """Half page-aligned ascending runs of 64 slots, half uniform slots.

    floor(length/2) rounded down to whole 64-slot runs come first, each run
    starting at a random page; the remaining ids are uniform."""
    n_runs = (length // 2) // PAGE
    pages = torch.randint(0, num_slots // PAGE, (n_runs,), generator=gen, dtype=torch.int64)
    runs = (pages[:, None] * PAGE + torch.arange(PAGE, dtype=torch.int64)[None, :]).reshape(-1)
    rest = torch.randint(0, num_slots, (length - runs.numel(),), generator=gen, dtype=torch.int64)
    return torch.cat([runs, rest]).to(torch.int32)


# ------------------------------------------------------------- workloads

def tiny_tp2(seed: int = 0, device="cpu", length: int = 64, fmt: str = "bf16") -> Workload:
    """bs=1, 12Q/1KV, pool [4096, 1, 256], `length` uniform slots with replacement."""
    num_slots = 4096
    kc, vc, ks, vs = make_pools(num_slots, 1, fmt, seed, device)
    g = _gen(seed, "cpu")
    sel = uniform_indices(length, num_slots, g)
    return Workload(make_query(1, 12, seed, device), kc, vc, sel.to(device),
                    cu_from_lengths([length]).to(device), fmt, ks, vs,
                    name=f"tiny_tp2_L{length}_{fmt}")


def tp1_mixed(seed: int = 1, device="cpu", bs: int = 16, num_slots: int = 262144,
              fmt: str = "bf16", max_len: int = MAX_CAPACITY, lengths=None) -> Workload:
    """bs sequences, 24Q/2KV, lengths ~ U[1, max_len], uniform slot ids."""
    kc, vc, ks, vs = make_pools(num_slots, 2, fmt, seed, device)
    g = _gen(seed, "cpu")
    if lengths is None:
        lengths = torch.randint(1, max_len + 1, (bs,), generator=g, dtype=torch.int64)
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    sel = uniform_indices(int(lengths.sum()), num_slots, g)
    return Workload(make_query(bs, 24, seed, device), kc, vc, sel.to(device),
                    cu_from_lengths(lengths).to(device), fmt, ks, vs,
                    capacity=max(int(lengths.max()), 1) if lengths.numel() else 1,
                    name=f"tp1_mixed_bs{bs}_{fmt}")


def tp1_saturated(seed: int = 2, device="cpu", bs: int = 128, num_slots: int = 1048576,
                  fmt: str = "bf16", length: int = MAX_CAPACITY, index_seed: Optional[int] = None,
                  pools=None) -> Workload:
    """bs sequences of exactly `length` slots: page-aligned 64-slot runs + uniform slots.

    `pools` may pass (k, v, k_scale, v_scale) already resident to build more
    index sets over the same pool; `index_seed` varies the index draw only."""
    if pools is None:
        pools = make_pools(num_slots, 2, fmt, seed, device)
    kc, vc, ks, vs = pools
    g = _gen(seed if index_seed is None else index_seed, "cpu")
    sel = torch.cat([runs_and_uniform_indices(length, kc.shape[0], g) for _ in range(bs)])
    return Workload(make_query(bs, 24, seed if index_seed is None else index_seed, device),
                    kc, vc, sel.to(device), cu_from_lengths([length] * bs).to(device), fmt, ks, vs,
                    capacity=length, name=f"tp1_saturated_bs{bs}_L{length}_{fmt}")


def tiered(seed: int = 4, device="cpu", bs: int = 16, num_slots: int = 16384,
           ring_slots: int = 4096, num_kv_heads: int = 2, lengths=None, max_len: int = MAX_CAPACITY,
           hot_share: float = 0.5, pools=None) -> Workload:
    """A tiered int8ring_int4 workload: each sequence's ids are a `hot_share` of
    slots that own their ring row (read from the int8_g64 ring) and uniform slots
    (mostly read from the int4_g32 pool), interleaved in a seeded order."""
    if pools is None:
        pools = make_tiered_pools(num_slots, num_kv_heads, ring_slots, seed, device)
    kc, vc, ks, vs, tier = pools
    g = _gen(seed, "cpu")
    if lengths is None:
        lengths = torch.randint(1, max_len + 1, (bs,), generator=g, dtype=torch.int64)
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    owner = tier["owner"].cpu().long()
    hot_slots = owner[owner >= 0]
    parts = []
    for L in lengths.tolist():
        nh = int(round(L * hot_share)) if hot_slots.numel() else 0
        hot = hot_slots[torch.randint(0, max(hot_slots.numel(), 1), (nh,), generator=g)]
        uni = torch.randint(0, kc.shape[0], (L - nh,), generator=g, dtype=torch.int64)
        ids = torch.cat([hot, uni])
        parts.append(ids[torch.randperm(L, generator=g)])
    sel = (torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64)).to(torch.int32)
    hq = 12 * num_kv_heads
    return Workload(make_query(bs, hq, seed, device), kc, vc, sel.to(device),
                    cu_from_lengths(lengths).to(device), TIERED, ks, vs,
                    capacity=max(int(lengths.max()), 1) if lengths.numel() else 1,
                    name=f"tiered_bs{bs}_R{ring_slots}", extra=dict(tier))


# ------------------------------------------- counter-based generator (replays)
#
# MurmurHash3's 32-bit finaliser (fmix32, A. Appleby, public domain) used as a
# counter-based generator: every value is a pure function of (seed, replay,
# b, j), so the same torch code regenerates a replay's lengths and slot ids
# on the GPU inside a captured graph and on the host for the oracle.

_M32 = 0xFFFFFFFF


def _mul32(h, c: int):
    """(h * c) mod 2^32 for h in [0, 2^32) (int or int64 tensor), without int64 overflow."""
    lo = h & 0xFFFF
    hi = h >> 16
    return (lo * c + (((hi * (c & 0xFFFF)) & 0xFFFF) << 16)) & _M32


def fmix32(h):
    """MurmurHash3 fmix32 of h in [0, 2^32); works on Python ints and int64 tensors."""
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def hash_key(seed: int, replay: torch.Tensor, b, j):
    """fmix32 chain over (seed, replay, b, j) -> int64 values in [0, 2^32).

    `seed` is a Python int; `replay`, `b`, `j` are int64 tensors (or ints)
    that broadcast; no host<->device traffic happens here."""
    h = fmix32((replay & _M32) ^ fmix32(int(seed) & _M32))
    h = fmix32(h ^ (b & _M32))
    return fmix32(h ^ ((j + 0x9E3779B9) & _M32))


BANDS = {"short": (1, 64), "medium": (512, 1024), "saturated": (MAX_CAPACITY, MAX_CAPACITY)}


def replay_lengths(seed: int, replay: torch.Tensor, bs: int, band: str, device) -> torch.Tensor:
    """int64 [bs] lengths of one replay, uniform in the band (inclusive)."""
    lo, hi = BANDS[band]
    b = torch.arange(bs, dtype=torch.int64, device=device)
    h = hash_key(seed, replay, b, -1)
    return lo + h % (hi - lo + 1)


def replay_inputs(seed: int, replay: torch.Tensor, bs: int, band: str, capacity: int,
                  num_slots: int, sel_out: torch.Tensor, cu_out: torch.Tensor) -> None:
    """Regenerate one replay's cu_seqlens and packed slot ids in place.

    Everything is torch tensor ops without host readback, so it can run inside
    a captured CUDA graph; `replay` is a 1-element int64 device tensor.
    `sel_out` holds bs*capacity ids; entries past cu[bs] are left stale."""
    dev = sel_out.device
    lens = replay_lengths(seed, replay, bs, band, dev)
    cu = torch.zeros(bs + 1, dtype=torch.int64, device=dev)
    cu[1:] = torch.cumsum(lens, 0)
    cu_out.copy_(cu.to(torch.int32))
    pos = torch.arange(bs * capacity, dtype=torch.int64, device=dev)
    b = torch.searchsorted(cu[1:], pos, right=True).clamp_(max=bs - 1)
    j = pos - cu[b]
    ids = hash_key(seed, replay, b, j) % num_slots
    live = pos < cu[bs]
    sel_out.copy_(torch.where(live, ids, torch.zeros_like(ids)).to(torch.int32))


# ----------------------------------------------------------- host subsets

def host_subset(w: Workload, rows) -> Workload:
    """Host workload holding only `rows` of a device workload, with the pool
    rows those sequences select copied to the host (slot ids remapped)."""
    rows = [int(r) for r in rows]
    cu = w.cu.cpu().long()
    sel = w.sel.cpu().long()
    parts = [sel[cu[b]:cu[b + 1]] for b in rows]
    flat = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.long)
    uniq, inv = torch.unique(flat, return_inverse=True)
    dev_idx = uniq.to(w.k_pool.device)
    k = w.k_pool.index_select(0, dev_idx).cpu()
    v = w.v_pool.index_select(0, dev_idx).cpu()
    if w.fmt == TIERED:
        return _tiered_subset(w, rows, cu, sel, uniq, inv)
    ks = vs = None
    if w.fmt in ("int8", "int4") or w.fmt in GROUPED:
        ks = w.k_scale.index_select(0, dev_idx).cpu()
        vs = w.v_scale.index_select(0, dev_idx).cpu()
    elif w.fmt == "fp8_e4m3":
        ks, vs = w.k_scale.cpu(), w.v_scale.cpu()
    lens = [int(cu[b + 1] - cu[b]) for b in rows]
    return Workload(w.q.cpu()[rows], k, v, inv.to(torch.int32), cu_from_lengths(lens), w.fmt,
                      ks, vs, w.softmax_scale, w.capacity, w.name + "_subset")


def _tiered_subset(w: Workload, rows, cu, sel, uniq, inv) -> Workload:
    """host_subset of a tiered workload: the selected slots become ids 0..n-1 of a
    tiered pool whose ring has one position per id (a power of two at least n), so
    id k owns ring row k exactly when its original slot owned its ring row."""
    tier = w.extra
    R = tier["owner"].shape[0]
    dev_idx = uniq.to(w.k_pool.device)
    pos = dev_idx & (R - 1)
    owner = tier["owner"].index_select(0, pos)
    hot = owner == dev_idx.to(owner.dtype)
    n = uniq.numel()
    R2 = 1
    while R2 < max(n, 1):
        R2 *= 2
    new_tier = {}
    for key in ("k_ring", "v_ring", "k_ring_scale", "v_ring_scale"):
        src = tier[key].index_select(0, pos)
        pad = torch.zeros((R2 - n,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
        new_tier[key] = torch.cat([src, pad]).cpu()
    new_owner = torch.full((R2,), -1, dtype=torch.int32)
    new_owner[:n] = torch.where(hot.cpu(), torch.arange(n, dtype=torch.int32),
                                torch.full((n,), -1, dtype=torch.int32))
    new_tier["owner"] = new_owner
    lens = [int(cu[b + 1] - cu[b]) for b in rows]
    return Workload(w.q.cpu()[rows], w.k_pool.index_select(0, dev_idx).cpu(),
                    w.v_pool.index_select(0, dev_idx).cpu(), inv.to(torch.int32),
                    cu_from_lengths(lens), w.fmt, w.k_scale.index_select(0, dev_idx).cpu(),
                    w.v_scale.index_select(0, dev_idx).cpu(), w.softmax_scale, w.capacity,
                    w.name + "_subset", new_tier)


# ------------------------------------------- compressed-block scores (top-k input)
#
# The top-k step takes one float32 score per compressed block of `ratio` tokens,
# produced upstream by a scoring step the pages do not define. These generators
# draw such scores: N(0,1) values with planted ties, -0.0 / +0.0, -inf and NaN, so
# the exact ranking rules are exercised; and context lengths that include the
# edge cases of the expansion (no block, whole blocks only, the longest tail).

TOPK_CAPACITY = 262144   # the pages' fixed 256K context capacity
TOPK_BUDGET = 2048       # token_topk (indexer budget)
TOPK_RATIO = 4           # compress ratio; row width 2048 + 4 - 1 = 2051


def topk_budget(ratio: int) -> int:
    """token_topk for a compress ratio: the pages' 2048, or the largest multiple of the
    ratio whose rows (token_topk + ratio - 1) still fit the decode's 2055 (2032 at 16)."""
    return min(TOPK_BUDGET, (MAX_CAPACITY - ratio + 1) // ratio * ratio)


def block_scores(bs: int, nblocks: int, seed: int, device="cpu", specials: bool = True) -> torch.Tensor:
    """float32 [bs, nblocks] N(0,1) block scores; with `specials`, about 1 % of the
    entries are replaced by repeats of a few shared values (ties), and a few by
    -0.0, +0.0, -inf and NaN."""
    g = _gen(seed, "cpu")
    s = torch.randn(bs, nblocks, generator=g, dtype=torch.float32)
    if specials:
        u = torch.rand(bs, nblocks, generator=g)
        shared = torch.tensor([0.5, 1.25, -0.75, 2.0], dtype=torch.float32)
        pick = torch.randint(0, 4, (bs, nblocks), generator=g)
        s = torch.where(u < 0.010, shared[pick], s)
        s = torch.where((u >= 0.010) & (u < 0.012), torch.full_like(s, -0.0), s)
        s = torch.where((u >= 0.012) & (u < 0.014), torch.zeros_like(s), s)
        s = torch.where((u >= 0.014) & (u < 0.016), torch.full_like(s, -float("inf")), s)
        s = torch.where((u >= 0.016) & (u < 0.018), torch.full_like(s, float("nan")), s)
    return s.to(device)


def context_lengths(bs: int, capacity: int, ratio: int, token_topk: int, seed: int) -> torch.Tensor:
    """int32 [bs] context lengths: uniform in [0, capacity], with the edge cases of
    the expansion placed first (empty, shorter than a block, exactly the kept
    blocks, the kept blocks plus the longest tail, one block more, the capacity)."""
    g = _gen(seed, "cpu")
    edge = [0, ratio - 1, ratio, token_topk, token_topk + ratio - 1, token_topk + ratio, capacity,
            capacity - 1]
    edge = [min(max(e, 0), capacity) for e in edge]
    lens = torch.randint(0, capacity + 1, (bs,), generator=g, dtype=torch.int64)
    for i, e in enumerate(edge[:bs]):
        lens[i] = e
    return lens.to(torch.int32)


def page_table(bs: int, capacity: int, page: int, seed: int, device="cpu") -> torch.Tensor:
    """int32 [bs, ceil(capacity / page)]: every sequence's pages are distinct
    physical pages of one shared pool, in a seeded random order."""
    g = _gen(seed, "cpu")
    npg = -(-capacity // page)
    perm = torch.randperm(bs * npg, generator=g, dtype=torch.int64)
    return perm.view(bs, npg).to(torch.int32).to(device)


def replay_block_scores(seed: int, replay: torch.Tensor, out: torch.Tensor) -> None:
    """Regenerate [bs, nblocks] block scores in place from the counter-based hash
    of (seed, replay, b, i), on the tensor's device (graph-capturable). The scores
    take 2^20 distinct values, so equal scores occur; hash values 0 and 1 mod 509
    give -0.0 and NaN."""
    bs, nb = out.shape
    dev = out.device
    b = torch.arange(bs, dtype=torch.int64, device=dev).view(-1, 1)
    i = torch.arange(nb, dtype=torch.int64, device=dev).view(1, -1)
    h = hash_key(seed, replay, b, i)
    v = ((h >> 12).to(torch.float32) - 524288.0) * (1.0 / 65536.0)
    v = torch.where(h % 509 == 0, torch.full_like(v, -0.0), v)
    v = torch.where(h % 509 == 1, torch.full_like(v, float("nan")), v)
    out.copy_(v)


def replay_context_lengths(seed: int, replay: torch.Tensor, capacity: int, out: torch.Tensor) -> None:
    """Regenerate int32 [bs] context lengths in [0, capacity] in place (graph-capturable)."""
    bs = out.shape[0]
    b = torch.arange(bs, dtype=torch.int64, device=out.device)
    out.copy_((hash_key(seed, replay, b, -7) % (capacity + 1)).to(torch.int32))
