"""Pins for the FP64 oracle: closed forms, library routines, brute force.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (dropped term, wrong sign, transposed operand, wrong
head mapping, swapped nibble, misplaced scale) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_paged_qsa_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_np(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _small_workload(fmt="bf16", bs=2, Hq=24, num_slots=512, lengths=(5, 9), seed=7):
    Hkv = Hq // 12
    kc, vc, ks, vs = I.make_pools(num_slots, Hkv, fmt, seed)
    q = I.make_query(bs, Hq, seed)
    g = torch.Generator().manual_seed(seed)
    sel = I.uniform_indices(int(sum(lengths)), num_slots, g)
    cu = I.cu_from_lengths(lengths)
    return I.Workload(q, kc, vc, sel, cu, fmt, ks, vs)


def _run(w, **kw):
    return oracle.decode(w.q, w.k_pool, w.v_pool, w.fmt, w.sel, w.cu, w.softmax_scale,
                         w.k_scale, w.v_scale, **kw)


# --------------------------------------------------------------- element decoders

def test_e4m3fn_decode_matches_torch_for_all_bytes():
    bytes_ = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = bytes_.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3fn_to_double(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3fn_golden_values():
    for line in open(os.path.join(GOLDEN, "e4m3fn_values.txt")):
        if line.startswith("#") or not line.strip():
            continue
        b, v = line.split()[:2]
        got = oracle.e4m3fn_to_double(int(b, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v)


def test_int4_nibbles_match_arithmetic_shift():
    for b in range(256):
        lo = int(np.int8(np.uint8((b << 4) & 0xFF).view(np.int8)) >> 4)
        hi = int(np.uint8(b).view(np.int8) >> 4)
        assert oracle.int4_value(b, 0) == lo
        assert oracle.int4_value(b, 1) == hi


def test_int4_packing_golden_and_quantiser_layout():
    pairs = []
    for line in open(os.path.join(GOLDEN, "int4_packing.txt")):
        if line.startswith("#") or not line.strip():
            continue
        e, o, byte = line.split()
        pairs.append((int(e), int(o), int(byte, 16)))
    for e, o, byte in pairs:
        assert oracle.int4_value(byte, 0) == e
        assert oracle.int4_value(byte, 1) == o
    # the input-side packer writes the same layout
    vals = torch.tensor([[v for e, o, _ in pairs for v in (e, o)]], dtype=torch.float32)
    # a row whose absmax is 8 with scale 8/7 would re-round; use exact codes instead
    codes = vals.to(torch.int8)
    lo = codes[..., 0::2].to(torch.int16) & 0xF
    hi = codes[..., 1::2].to(torch.int16) & 0xF
    packed = (lo | (hi << 4)).to(torch.uint8)
    assert packed.tolist()[0] == [b for _, _, b in pairs]


def test_bf16_to_double_matches_torch():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 1 << 16, (4000,), generator=g, dtype=torch.int32)
    t = bits.to(torch.int16).view(torch.bfloat16)
    ref = t.to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b) & 0xFFFF) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(ref[fin], got[fin])


def test_round_bf16_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(20000, generator=g) * 20)
    # ties: values exactly halfway between two bf16 neighbours
    base = torch.randn(2000, generator=g).to(torch.bfloat16).to(torch.float32)
    half_ulp = torch.ldexp(torch.ones_like(base), torch.frexp(base)[1] - 9)
    x = torch.cat([x, base + half_ulp, base - half_ulp, torch.tensor([1e-40, -3e-39, 0.0])])
    ref = _bf16_np(x.to(torch.bfloat16))
    got = oracle.round_bf16_bits(x.to(torch.float64).numpy())
    assert np.array_equal(ref, got)


def test_round_bf16_ties_to_even_closed_form():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert oracle.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 lies halfway between 1+2^-7 and 1+2^-6: even is 1+2^-6
    assert oracle.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    # a double that is not a float32 value: 1 + 2^-8 + 2^-40 rounds up
    assert oracle.round_bf16(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == 1 + 2 ** -7


# ------------------------------------------------------------- dequantisation

@pytest.mark.parametrize("fmt", ["fp8_e4m3", "int8", "int4"])
def test_dequant_within_half_quantum_of_source(fmt):
    """dequant(quantise(x)) stays within the format's rounding bound of x."""
    x = I.normal_values((64, 2, 256), 11)
    codes, s = I.quantize_pool(x, fmt)
    for g in range(2):
        xr = oracle.dequant_rows(codes, fmt, range(64), g, s)
        err = np.abs(xr - x[:, g].double().numpy())
        if fmt == "fp8_e4m3":
            # e4m3 keeps 3 mantissa bits: half an ulp is 2^-4 of the value's
            # binade; below 2^-6 * s the spacing is the subnormal step 2^-9 * s
            y = np.abs(x[:, g].double().numpy())
            bound = np.maximum(y * 2.0 ** -4, 2.0 ** -10 * float(s[0])) * (1 + 1e-6)
        else:
            bound = 0.5 * s[:, g].double().numpy()[:, None] * (1 + 1e-6)
        assert (err <= bound + 1e-12).all()


def test_quant_error_bands_from_the_pages():
    """Relative RMS error bands (sglang PR #37798, "Accuracy Tests"): e4m3 in
    (1 %, 4 %) on N(0, 3); int8 below 1.2 %. The int4 band 8-11.5 % is for
    32-channel groups; with one scale per 256-channel row the error is larger,
    and the reading used here is (8 %, 14 %)."""
    def rel_rms(fmt, std):
        x = I.normal_values((256, 2, 256), 12, std=std)
        codes, s = I.quantize_pool(x, fmt)
        xr = np.stack([oracle.dequant_rows(codes, fmt, range(256), g, s) for g in range(2)], 1)
        xd = x.double().numpy()
        return math.sqrt(((xr - xd) ** 2).mean() / (xd ** 2).mean())

    assert 0.01 < rel_rms("fp8_e4m3", 3.0) < 0.04
    assert rel_rms("int8", 1.0) < 0.012
    assert 0.08 < rel_rms("int4", 1.0) < 0.14


def test_scale_is_per_slot_and_kv_head():
    """With power-of-two scales, int8 codes * s are exact bf16 values, so the
    int8 oracle must equal the bf16 oracle run on those values exactly."""
    num_slots, Hkv = 64, 2
    g = torch.Generator().manual_seed(5)
    codes_k = torch.randint(-127, 128, (num_slots, Hkv, 256), generator=g).to(torch.int8)
    codes_v = torch.randint(-127, 128, (num_slots, Hkv, 256), generator=g).to(torch.int8)
    e = torch.arange(num_slots * Hkv).reshape(num_slots, Hkv)
    sk = torch.ldexp(torch.ones(num_slots, Hkv), -(e % 5) - 3).float()
    sv = torch.ldexp(torch.ones(num_slots, Hkv), -(e % 7) - 2).float()
    kb = (codes_k.float() * sk[..., None]).to(torch.bfloat16)
    vb = (codes_v.float() * sv[..., None]).to(torch.bfloat16)
    assert torch.equal(kb.float(), codes_k.float() * sk[..., None])
    q = I.make_query(3, 24, 5)
    sel = I.uniform_indices(40, num_slots, g)
    cu = I.cu_from_lengths([10, 17, 13])
    a = oracle.decode(q, codes_k, codes_v, "int8", sel, cu, 1 / 16, sk, sv)
    b = oracle.decode(q, kb, vb, "bf16", sel, cu, 1 / 16)
    assert np.array_equal(a, b)


# -------------------------------------------------------------------- decode

@pytest.mark.parametrize("fmt", I.FORMATS)
def test_single_index_returns_that_v_row(fmt):
    w = _small_workload(fmt, lengths=(1, 1))
    out = _run(w)
    for b in range(2):
        slot = int(w.sel[b])
        for h in range(24):
            gkv = h // 12
            if fmt == "bf16":
                ref = w.v_pool[slot, gkv].to(torch.float64).numpy()
            elif fmt == "fp8_e4m3":
                ref = (w.v_pool[slot, gkv].view(torch.float8_e4m3fn).to(torch.float64)
                       * float(w.v_scale[0])).numpy()
            elif fmt == "int8":
                ref = (w.v_pool[slot, gkv].to(torch.float64) * float(w.v_scale[slot, gkv])).numpy()
            elif fmt == "int8_g64":
                sc = w.v_scale[slot, gkv].to(torch.float64).repeat_interleave(64)
                ref = (w.v_pool[slot, gkv].to(torch.float64) * sc).numpy()
            elif fmt == "int4_g32":
                byts = w.v_pool[slot, gkv].numpy().astype(np.int64)
                vals = np.stack([(byts & 0xF) - 8, (byts >> 4) - 8], 1).reshape(-1)
                sc = w.v_scale[slot, gkv].to(torch.float64).repeat_interleave(32).numpy()
                ref = vals * sc
            else:
                byts = w.v_pool[slot, gkv].numpy()
                lo = (byts.astype(np.int16) << 12).astype(np.int16) >> 12
                hi = (byts.astype(np.int16) << 8).astype(np.int16) >> 12
                ref = np.stack([lo, hi], 1).reshape(-1) * float(w.v_scale[slot, gkv])
            assert np.array_equal(out[b, h], ref)


def test_identical_keys_give_mean_of_selected_values():
    w = _small_workload("bf16", lengths=(7, 12))
    # every selected slot gets the same K row, so the softmax is uniform
    k = w.k_pool.clone()
    k[w.sel.long()] = k[0].clone()
    out = oracle.decode(w.q, k, w.v_pool, "bf16", w.sel, w.cu, w.softmax_scale)
    for b in range(2):
        ids = w.sel[w.cu[b]:w.cu[b + 1]].long()
        for h in range(24):
            ref = w.v_pool[ids, h // 12].to(torch.float64).mean(0).numpy()
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-14)


def test_duplicates_weigh_by_multiplicity():
    """[a, a, b] is a two-row softmax with logit s_a + ln 2: o = sigma(t) Va + (1 - sigma(t)) Vb."""
    w = _small_workload("bf16", bs=1, lengths=(3,))
    a, bslot = 17, 301
    sel = torch.tensor([a, a, bslot], dtype=torch.int32)
    out = oracle.decode(w.q, w.k_pool, w.v_pool, "bf16", sel, w.cu, w.softmax_scale)
    for h in range(24):
        gkv = h // 12
        q = w.q[0, h].double()
        sa = float(q @ w.k_pool[a, gkv].double()) / 16
        sb = float(q @ w.k_pool[bslot, gkv].double()) / 16
        t = sa + math.log(2.0) - sb
        wa = 1.0 / (1.0 + math.exp(-t))
        ref = wa * w.v_pool[a, gkv].double() + (1 - wa) * w.v_pool[bslot, gkv].double()
        np.testing.assert_allclose(out[0, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_permutation_invariance():
    w = _small_workload("int8", bs=1, lengths=(50,))
    out = _run(w)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(9))
    out2 = oracle.decode(w.q, w.k_pool, w.v_pool, "int8", w.sel[perm], w.cu, w.softmax_scale,
                         w.k_scale, w.v_scale)
    np.testing.assert_allclose(out, out2, rtol=1e-12, atol=1e-14)


def test_peaked_scores_select_the_argmax_row():
    w = _small_workload("bf16", bs=1, lengths=(40,))
    q = (w.q.float() * 64).to(torch.bfloat16)
    out = oracle.decode(q, w.k_pool, w.v_pool, "bf16", w.sel, w.cu, 1 / 16)
    ids = w.sel.long()
    for h in range(24):
        gkv = h // 12
        s = w.k_pool[ids, gkv].double() @ q[0, h].double()
        top2 = torch.topk(s, 2).values
        if float(top2[0] - top2[1]) / 16 < 40:
            continue
        ref = w.v_pool[ids[int(torch.argmax(s))], gkv].double().numpy()
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Hq", [12, 24])
def test_contiguous_selection_equals_sdpa(Hq):
    """Selecting slots 0..L-1 in order reduces to dense attention: torch's
    scaled_dot_product_attention in float64 with the KV heads expanded by GQA."""
    Hkv = Hq // 12
    L = 37
    kc, vc, _, _ = I.make_pools(64, Hkv, "bf16", 13)
    q = I.make_query(1, Hq, 13)
    sel = torch.arange(L, dtype=torch.int32)
    out = oracle.decode(q, kc, vc, "bf16", sel, I.cu_from_lengths([L]), 1 / 16)
    kk = kc[:L].double().permute(1, 0, 2).repeat_interleave(12, 0)   # [Hq, L, D]
    vv = vc[:L].double().permute(1, 0, 2).repeat_interleave(12, 0)
    qq = q[0].double()[:, None, :]                                    # [Hq, 1, D]
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=1 / 16)[:, 0]
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_brute_force_pure_python_tiny():
    w = _small_workload("bf16", bs=2, Hq=12, num_slots=32, lengths=(3, 4), seed=21)
    out = _run(w)
    qf = w.q.double().tolist()
    kf = w.k_pool.double().tolist()
    vf = w.v_pool.double().tolist()
    for b in range(2):
        ids = w.sel[w.cu[b]:w.cu[b + 1]].tolist()
        for h in range(12):
            s = [sum(qf[b][h][d] * kf[i][0][d] for d in range(256)) / 16 for i in ids]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            for d in range(0, 256, 17):
                ref = math.fsum(e[j] * vf[ids[j]][0][d] for j in range(len(ids))) / z
                assert abs(out[b, h, d] - ref) <= 1e-13 * (1 + abs(ref))


def test_empty_selection_gives_zeros_and_rows_subset():
    w = _small_workload("fp8_e4m3", bs=4, lengths=(6, 0, 11, 0))
    out = _run(w)
    assert not out[1].any() and not out[3].any()
    assert out[0].any() and out[2].any()
    sub = _run(w, rows=[2, 0])
    assert np.array_equal(sub[0], out[2]) and np.array_equal(sub[1], out[0])


def test_refuses_inputs_outside_the_contract():
    w = _small_workload("bf16", lengths=(3, 4))
    bad = w.sel.clone()
    bad[2] = w.num_slots
    with pytest.raises(oracle.OracleRefused):
        oracle.decode(w.q, w.k_pool, w.v_pool, "bf16", bad, w.cu, 1 / 16)
    cu = w.cu.clone()
    cu[1] = 5
    cu[2] = 4
    with pytest.raises(oracle.OracleRefused):
        oracle.decode(w.q, w.k_pool, w.v_pool, "bf16", w.sel, cu, 1 / 16)


def test_thread_count_does_not_change_results():
    w = _small_workload("int4", bs=3, lengths=(30, 1, 64))
    a = _run(w, threads=1)
    b = _run(w, threads=4)
    assert np.array_equal(a, b)


# ---------------------------------------------------------- quantising KV write

def test_e4m3fn_encode_matches_torch_cast_and_saturates():
    g = torch.Generator().manual_seed(21)
    x = torch.randn(50000, generator=g) * torch.exp(torch.randn(50000, generator=g) * 3)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11])])
    inside = x.clamp(-448, 448)
    ref = inside.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3fn_encode(float(v)) for v in inside])
    assert np.array_equal(ref, got)
    # beyond the largest finite value the write saturates (the cast alone would give NaN)
    for v, code in ((449.0, 0x7E), (1e6, 0x7E), (-500.0, 0xFE), (float("inf"), 0x7E)):
        assert oracle.e4m3fn_encode(v) == code
    assert oracle.e4m3fn_encode(float("nan")) == 0x7F


@pytest.mark.parametrize("fmt", ["int8", "int4", "fp8_e4m3"])
def test_quantize_rows_matches_the_torch_quantiser(fmt):
    """Two independent implementations of the write-side quantiser agree bit for bit."""
    x = I.normal_values((300, 1, 256), 22).to(torch.bfloat16)
    xf = x.float()
    codes_t, s_t = I.quantize_pool(xf, fmt)
    scale = float(s_t[0]) if fmt == "fp8_e4m3" else 1.0
    codes, scales = oracle.quantize_rows(x[:, 0], fmt, fp8_scale=scale)
    assert np.array_equal(codes.view(np.uint8), codes_t[:, 0].view(torch.uint8).numpy())
    if fmt != "fp8_e4m3":
        assert np.array_equal(scales, s_t[:, 0].numpy())


def test_quantize_rows_ties_zero_rows_and_clamps():
    # absmax 127 -> scale exactly 1; halves round to even
    row = torch.zeros(256)
    row[0], row[1], row[2], row[3], row[4] = 127.0, 2.5, 3.5, -2.5, 100.5
    zero = torch.zeros(256)
    x = torch.stack([row, zero]).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows(x, "int8")
    assert scales[0] == 1.0 and scales[1] == 0.0
    assert codes[0, :5].tolist() == [127, 2, 4, -2, 100]
    assert not codes[1].any()
    # int4: absmax 7 -> scale 1; channel 2i in the low nibble; halves to even
    row4 = torch.zeros(256)
    row4[0], row4[1], row4[2], row4[3] = 7.0, -3.5, 2.5, 0.5
    c4, s4 = oracle.quantize_rows(row4[None].to(torch.bfloat16), "int4")
    assert s4[0] == 1.0
    assert c4[0, 0] == 0xC7 and c4[0, 1] == 0x02 and not c4[0, 2:].any()


def test_quantize_then_dequantize_round_trip():
    x = I.normal_values((64, 1, 256), 23, std=2.0).to(torch.bfloat16)
    xd = x[:, 0].double().numpy()
    for fmt, qmax in (("int8", 127), ("int4", 7)):
        codes, scales = oracle.quantize_rows(x[:, 0], fmt)
        pool = torch.from_numpy(codes.view(np.uint8) if fmt == "int4" else codes)[:, None]
        back = oracle.dequant_rows(pool, fmt, range(64), 0, torch.from_numpy(scales)[:, None])
        # |rint(fl(x / s)) - x / s| <= 1/2 + |fl(x / s) - x / s|, the second term below qmax * 2^-24
        assert (np.abs(back - xd) <= (0.5 + qmax * 2.0 ** -23) * scales[:, None]).all()


# ------------------------------------------------------- grouped pool formats

def _golden_grouped():
    nib, groups, clamp = [], {}, None
    for line in open(os.path.join(GOLDEN, "grouped_formats.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "nibble":
            nib.append((int(f[1], 16), int(f[2]), int(f[3])))
        elif f[0] == "group":
            pairs = [(int(f[i + 1]), int(f[i + 3])) for i in range(3, len(f), 4)]
            groups[f[1]] = (int(f[2]), pairs)
        elif f[0] == "clamp":
            clamp = float(f[1])
    return nib, groups, clamp


def test_fp16_decode_matches_numpy_for_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])


def test_round_fp16_matches_numpy_including_ties_and_overflow():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000)).astype(np.float32)
    base = rng.standard_normal(2000).astype(np.float16).astype(np.float32)
    m, e = np.frexp(base)
    half_ulp = np.ldexp(np.ones_like(base), e - 12).astype(np.float32)  # ties between neighbours
    edges = np.array([65504, 65519.996, 65520, 70000, 2.0 ** -14, 2.0 ** -24, 2.0 ** -25,
                      3 * 2.0 ** -25, 1e-9, 0.0, -0.0], dtype=np.float32)
    x = np.concatenate([x, base + half_ulp, base - half_ulp, edges, -edges])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.round_fp16_bits(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # closed forms: 1 + 2^-11 is halfway between 1 and 1 + 2^-10 -> 1 (even)
    assert oracle.round_fp16_bits(1 + 2 ** -11) == 0x3C00
    assert oracle.round_fp16_bits(1 + 3 * 2 ** -11) == 0x3C02


def test_grouped_golden_nibbles_groups_and_clamp():
    nib, groups, clamp = _golden_grouped()
    for byte, even, odd in nib:
        assert oracle.int4_offset_value(byte, 0) == even
        assert oracle.int4_offset_value(byte, 1) == odd
    for fmt, (size, pairs) in groups.items():
        # codes 1 everywhere, scale of group k = 2^k: a channel reads its group's scale
        G = 256 // size
        codes = torch.full((1, 1, 128 if fmt == "int4_g32" else 256),
                           0x99 if fmt == "int4_g32" else 1, dtype=torch.uint8)
        if fmt == "int8_g64":
            codes = codes.view(torch.int8)
        sc = torch.tensor([[[2.0 ** k for k in range(G)]]], dtype=torch.float16)
        row = oracle.dequant_rows(codes, fmt, [0], 0, sc)[0]
        assert oracle.GROUP[fmt] == size
        for ch, grp in pairs:
            assert row[ch] == 2.0 ** grp
    for fmt in ("int8_g64", "int4_g32"):
        x = torch.zeros(1, 256)
        x[0, 0] = 3.0e38  # absmax / q far above the binary16 range
        x[0, 1] = -1.0e10
        _, s = oracle.quantize_rows(x.to(torch.bfloat16), fmt)
        assert float(s[0, 0]) == clamp and float(s[0, 1]) == 0.0


@pytest.mark.parametrize("fmt", ["int8_g64", "int4_g32"])
def test_grouped_decode_equals_bf16_pool_with_the_same_values(fmt):
    """Codes times power-of-two binary16 scales are exact bf16 values: decoding the
    grouped pool must equal decoding a bf16 pool that holds those values."""
    gs = oracle.GROUP[fmt]
    slots, Hkv, G = 64, 2, 256 // gs
    g = torch.Generator().manual_seed(31)
    if fmt == "int8_g64":
        codes = torch.randint(-127, 128, (2, slots, Hkv, 256), generator=g)
        packed = codes.to(torch.int8)
    else:
        codes = torch.randint(-7, 8, (2, slots, Hkv, 256), generator=g)
        u = (codes + 8).to(torch.int16)
        packed = (u[..., 0::2] | (u[..., 1::2] << 4)).to(torch.uint8)
    exps = torch.randint(-6, 4, (2, slots, Hkv, G), generator=g).to(torch.float32)
    scales = torch.pow(2.0, exps).to(torch.float16)
    values = codes.to(torch.float64) * scales.to(torch.float64).repeat_interleave(gs, -1)
    bf = values.to(torch.bfloat16)
    assert torch.equal(bf.to(torch.float64), values)
    q = I.make_query(3, 12 * Hkv, 32)
    sel = I.uniform_indices(3 * 40, slots, g)
    cu = I.cu_from_lengths([40, 40, 40])
    got = oracle.decode(q, packed[0], packed[1], fmt, sel, cu, 1 / 16, scales[0], scales[1])
    ref = oracle.decode(q, bf[0], bf[1], "bf16", sel, cu, 1 / 16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", ["int8_g64", "int4_g32"])
def test_grouped_quantisers_agree_and_round_trip(fmt):
    """The oracle's write-side quantiser and the input generator's torch one agree
    bit for bit, and dequant(quantise(x)) is within half a step of x."""
    x = I.normal_values((200, 1, 256), 33, std=3.0).to(torch.bfloat16)
    x[0] = 0.0
    x[1, 0, :40] = 0.0           # an all-zero group
    x[2, 0, 5] = 2.0e9           # a group whose scale clamps
    codes, scales = oracle.quantize_rows(x[:, 0], fmt)
    codes_t, s_t = I.quantize_pool(x.float(), fmt)
    assert np.array_equal(codes.view(np.uint8), codes_t[:, 0].view(torch.uint8).numpy())
    assert np.array_equal(scales.view(np.uint16), s_t[:, 0].view(torch.int16).numpy().view(np.uint16))
    back = oracle.dequant_rows(torch.from_numpy(codes.view(np.uint8) if fmt == "int4_g32" else codes)[:, None],
                               fmt, range(200), 0, torch.from_numpy(scales)[:, None])
    xd = x[:, 0].double().numpy()
    s = scales.astype(np.float64).repeat(oracle.GROUP[fmt], -1)
    qmax = 127 if fmt == "int8_g64" else 7
    ok = np.ones_like(xd, dtype=bool)
    ok[2] = False  # the clamped group saturates
    assert (np.abs(back - xd)[ok] <= ((0.5 + qmax * 2.0 ** -23) * s)[ok]).all()
    assert back[2, 5] == qmax * 65504.0


def test_grouped_error_bands_from_the_pages():
    """Relative RMS error bands of the pages' pool tests (sglang PR #37798, "Accuracy
    Tests"): int8 with 64-channel groups below 1.2 %, int4 with 32-channel groups in
    8-11.5 %; measured on N(0, 1) draws."""
    def rel_rms(fmt):
        x = I.normal_values((256, 2, 256), 34)
        codes, s = I.quantize_pool(x, fmt)
        xr = np.stack([oracle.dequant_rows(codes, fmt, range(256), g, s) for g in range(2)], 1)
        xd = x.double().numpy()
        return math.sqrt(((xr - xd) ** 2).mean() / (xd ** 2).mean())

    assert rel_rms("int8_g64") < 0.012
    assert 0.08 < rel_rms("int4_g32") < 0.115


def test_grouped_quantiser_ties_and_zero_groups():
    row = torch.zeros(256)
    row[0], row[1], row[2], row[3] = 127.0, 2.5, 3.5, -2.5     # group 0: s16 = 1
    row[64], row[65] = 7.0, 0.5                                 # group 1: s16 = 7/127 rounded
    codes, s = oracle.quantize_rows(row[None].to(torch.bfloat16), "int8_g64")
    assert float(s[0, 0]) == 1.0 and codes[0, :4].tolist() == [127, 2, 4, -2]
    assert float(s[0, 2]) == 0.0 and not codes[0, 128:].any()
    s1 = np.float16(np.float32(7.0) / np.float32(127.0))
    assert s[0, 1] == s1 and codes[0, 64] == np.rint(np.float32(7.0) / np.float32(s1))
    row4 = torch.zeros(256)
    row4[0], row4[1], row4[2], row4[3] = 7.0, -3.5, 2.5, 0.5    # group 0: s16 = 1
    c4, s4 = oracle.quantize_rows(row4[None].to(torch.bfloat16), "int4_g32")
    assert float(s4[0, 0]) == 1.0
    # offset binary, even channel low: (7 + 8, -4 + 8) -> 0x4f; (2 + 8, 0 + 8) -> 0x8a
    assert c4[0, 0] == 0x4F and c4[0, 1] == 0x8A
    assert (c4[0, 2:] == 0x88).all()                            # zero codes read 8


# ------------------------------------------------ tiered int8ring_int4 pools

def _tiered_run(w, owner=None, **kw):
    t = w.extra
    return oracle.decode_tiered(w.q, w.k_pool, w.v_pool, w.sel, w.cu, w.softmax_scale, w.k_scale,
                                w.v_scale, t["k_ring"], t["v_ring"], t["k_ring_scale"],
                                t["v_ring_scale"], t["owner"] if owner is None else owner, **kw)


def test_tiered_all_hot_is_int8_g64_and_all_cold_is_int4_g32():
    """The pages' tiered tests: all-hot equals the int8 kernel, all-cold the int4 one;
    a stale owner (another slot of the same ring row) reads the int4 row."""
    slots, R = 1024, 1024
    w = I.tiered(seed=40, bs=3, num_slots=slots, ring_slots=R, lengths=[7, 300, 64])
    t = w.extra
    all_hot = torch.arange(R, dtype=torch.int32)
    # owner[p] = p with R = slots: every slot is hot and its ring row is ring[slot]
    hot = _tiered_run(w, owner=all_hot)
    ref8 = oracle.decode(w.q, t["k_ring"], t["v_ring"], "int8_g64", w.sel, w.cu, w.softmax_scale,
                         t["k_ring_scale"], t["v_ring_scale"])
    assert np.array_equal(hot, ref8)
    cold = _tiered_run(w, owner=torch.full((R,), -1, dtype=torch.int32))
    ref4 = oracle.decode(w.q, w.k_pool, w.v_pool, "int4_g32", w.sel, w.cu, w.softmax_scale,
                         w.k_scale, w.v_scale)
    assert np.array_equal(cold, ref4)
    stale = _tiered_run(w, owner=all_hot + R)          # same positions, other slots
    assert np.array_equal(stale, ref4)


def test_tiered_reads_the_ring_row_exactly_when_the_owner_matches():
    """Exact values (power-of-two scales, small codes) in both tiers: the tiered
    decode equals a bf16 pool holding, per slot, the ring value when
    owner[slot & (R-1)] == slot and the int4_g32 value otherwise."""
    slots, R, Hkv = 512, 128, 2
    g = torch.Generator().manual_seed(41)
    c8 = torch.randint(-127, 128, (2, R, Hkv, 256), generator=g)
    c4 = torch.randint(-7, 8, (2, slots, Hkv, 256), generator=g)
    s8 = torch.pow(2.0, torch.randint(-5, 3, (2, R, Hkv, 4), generator=g).float()).to(torch.float16)
    s4 = torch.pow(2.0, torch.randint(-5, 3, (2, slots, Hkv, 8), generator=g).float()).to(torch.float16)
    owner = torch.randint(-1, slots, (R,), generator=g).to(torch.int32)
    owner[::3] = (torch.arange(R, dtype=torch.int32) + R * torch.randint(0, slots // R, (R,), generator=g).to(torch.int32))[::3]
    u = (c4 + 8).to(torch.int16)
    packed4 = (u[..., 0::2] | (u[..., 1::2] << 4)).to(torch.uint8)
    v8 = c8.double() * s8.double().repeat_interleave(64, -1)
    v4 = c4.double() * s4.double().repeat_interleave(32, -1)
    sl = torch.arange(slots)
    is_hot = owner.long()[sl & (R - 1)] == sl
    assert 0 < int(is_hot.sum()) < slots
    vals = torch.where(is_hot.view(1, -1, 1, 1), v8[:, sl & (R - 1)], v4)
    bf = vals.to(torch.bfloat16)
    assert torch.equal(bf.double(), vals)
    q = I.make_query(2, 12 * Hkv, 42)
    sel = torch.randint(0, slots, (2 * 200,), generator=g).to(torch.int32)
    cu = I.cu_from_lengths([200, 200])
    got = oracle.decode_tiered(q, packed4[0], packed4[1], sel, cu, 1 / 16, s4[0], s4[1],
                               c8[0].to(torch.int8), c8[1].to(torch.int8), s8[0], s8[1], owner)
    ref = oracle.decode(q, bf[0], bf[1], "bf16", sel, cu, 1 / 16)
    assert np.array_equal(got, ref)


def test_tiered_write_in_token_order_with_ring_wrap_and_collisions():
    """R = 64 over 4096 slots (the pages' ring-wrap test): after a write of 500
    tokens, each touched ring row belongs to the last token of the write with that
    ring position, holds that token's int8_g64 row, and every written slot holds its
    int4_g32 row; untouched ring rows and slots keep their contents."""
    slots, R, Hkv, n = 4096, 64, 2, 500
    g = torch.Generator().manual_seed(43)
    pools = {
        "k_pool": np.full((slots, Hkv, 128), 0x5A, np.uint8), "v_pool": np.full((slots, Hkv, 128), 0xA5, np.uint8),
        "k_scale": np.full((slots, Hkv, 8), 3.0, np.float16), "v_scale": np.full((slots, Hkv, 8), 5.0, np.float16),
        "k_ring": np.full((R, Hkv, 256), 9, np.int8), "v_ring": np.full((R, Hkv, 256), -9, np.int8),
        "k_ring_scale": np.full((R, Hkv, 4), 7.0, np.float16), "v_ring_scale": np.full((R, Hkv, 4), 11.0, np.float16),
        "owner": np.full(R, -1, np.int32),
    }
    sl = torch.randperm(slots, generator=g)[:n].to(torch.int32)   # 500 slots over 64 ring rows
    xk = I.normal_values((n, Hkv, 256), 44).to(torch.bfloat16)
    xv = I.normal_values((n, Hkv, 256), 45).to(torch.bfloat16)
    before = {k: v.copy() for k, v in pools.items()}
    oracle.write_tiered(xk, xv, sl, pools)
    c8k, s8k = oracle.quantize_rows(xk.reshape(n * Hkv, 256), "int8_g64")
    c4k, s4k = oracle.quantize_rows(xk.reshape(n * Hkv, 256), "int4_g32")
    last = {}
    for i, s in enumerate(sl.tolist()):
        last[s % R] = i                                  # the later token wins
    for p in range(R):
        if p in last:
            i = last[p]
            assert pools["owner"][p] == sl[i]
            assert np.array_equal(pools["k_ring"][p], c8k.reshape(n, Hkv, 256)[i])
            assert np.array_equal(pools["k_ring_scale"][p], s8k.reshape(n, Hkv, 4)[i])
        else:
            assert pools["owner"][p] == -1 and np.array_equal(pools["k_ring"][p], before["k_ring"][p])
    for i, s in enumerate(sl.tolist()):
        assert np.array_equal(pools["k_pool"][s], c4k.reshape(n, Hkv, 128)[i])
        assert np.array_equal(pools["k_scale"][s], s4k.reshape(n, Hkv, 8)[i])
    untouched = np.setdiff1d(np.arange(slots), sl.numpy())
    assert np.array_equal(pools["v_pool"][untouched], before["v_pool"][untouched])
    assert len(last) < n                                  # collisions happened
