"""FP64 CPU oracle for packed QSA decode.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the product package never imports
it, and it imports nothing from the product package. The arithmetic lives in
``qsa_oracle.c`` (plain C, FP64, OpenMP over (sequence, head)); this module
only marshals arrays into it.

Definition followed (sglang PR #36845, "Changes" / "Optimized kernel";
sglang PR #37798, "Modifications"; 1Cat-vLLM PR #523, "Purpose"): for each
sequence b and query head h with KV head g = h // (Hq // Hkv),
``o = softmax(scale * q . Khat[I]^T) @ Vhat[I]`` over the selected slots
``I = sel[cu[b]:cu[b+1]]`` in order, duplicates kept; an empty selection
gives zeros. Khat/Vhat are the exactly dequantised pool rows.

It also holds the quantising KV write (``quantize_rows``): the codes and
scales the pools' write path produces, in binary32; and the tiered
``int8ring_int4`` pool (``decode_tiered``, ``write_tiered``; sglang PR #37798,
"Modifications", the tiered KV pool module): every token is written as an
int4_g32 row of its slot and as an int8_g64 row of the ring position
``slot & (R - 1)``, whose owner entry becomes the slot; a reader takes the ring
row when ``owner[slot & (R - 1)] == slot`` and the int4_g32 row otherwise.

Pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, library routines and brute force (see that file).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FORMATS = {"bf16": 0, "fp8_e4m3": 1, "int8": 2, "int4": 3, "int8_g64": 4, "int4_g32": 5}
GROUP = {"int8_g64": 64, "int4_g32": 32}     # channels per binary16 scale
NIBBLE = ("int4", "int4_g32")              # two 4-bit codes per byte

_lib = None


def build(force: bool = False) -> str:
    """Compile qsa_oracle.c into liboracle.so with gcc (IEEE FP64, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    lib.orc_bf16_to_double.restype = ctypes.c_double
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_e4m3fn_to_double.restype = ctypes.c_double
    lib.orc_e4m3fn_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_int4_value.restype = ctypes.c_int
    lib.orc_int4_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.orc_fp16_to_double.restype = ctypes.c_double
    lib.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_round_fp16.restype = ctypes.c_uint16
    lib.orc_round_fp16.argtypes = [ctypes.c_float]
    lib.orc_int4_offset_value.restype = ctypes.c_int
    lib.orc_int4_offset_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.orc_round_bf16.restype = ctypes.c_uint16
    lib.orc_round_bf16.argtypes = [ctypes.c_double]
    lib.orc_round_bf16_array.restype = None
    lib.orc_round_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.orc_dequant_row.restype = None
    lib.orc_dequant_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    lib.orc_decode.restype = ctypes.c_int
    lib.orc_decode.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,          # q, q_sb, q_sh
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,           # k_pool, v_pool, format
        ctypes.c_int64, ctypes.c_int, ctypes.c_int,               # num_slots, Hkv, D
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,        # k_scale, v_scale, scale
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,         # sel, n_sel, cu
        ctypes.c_int, ctypes.c_int,                               # bs, Hq
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,  # rows, n_rows, out, threads
    ]
    lib.orc_decode_tiered.restype = ctypes.c_int
    lib.orc_decode_tiered.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,          # q, q_sb, q_sh
        ctypes.c_void_p, ctypes.c_void_p,                         # k_pool, v_pool (int4_g32)
        ctypes.c_int64, ctypes.c_int, ctypes.c_int,               # num_slots, Hkv, D
        ctypes.c_void_p, ctypes.c_void_p,                         # k_scale, v_scale
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # rings + scales
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_double,         # owner, R, scale
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,         # sel, n_sel, cu
        ctypes.c_int, ctypes.c_int,                               # bs, Hq
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,  # rows, n_rows, out, threads
    ]
    lib.orc_max_threads.restype = ctypes.c_int
    lib.orc_e4m3fn_encode.restype = ctypes.c_uint8
    lib.orc_e4m3fn_encode.argtypes = [ctypes.c_float]
    lib.orc_quantize_rows.restype = ctypes.c_int
    lib.orc_quantize_rows.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    _lib = lib
    return lib


class OracleRefused(ValueError):
    """The input breaks the decode contract (bad cu_seqlens or slot ids)."""


def _np(a, dtype=None):
    """Contiguous host numpy view of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):
        import torch

        t = a.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must be host tensors")
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16).view(torch.uint16) if hasattr(torch, "uint16") else t.view(torch.int16)
        elif t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        elif t.dtype == torch.float16:
            t = t.view(torch.int16)
        a = t.contiguous().numpy()
        if a.dtype == np.int16:
            a = a.view(np.uint16)
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        a = a.astype(dtype)
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _scales(a, fmt: str):
    """Scales as the C side reads them: float32, or binary16 bits for the grouped formats."""
    if a is None:
        return None
    if fmt in GROUP:
        n = _np(a)
        if n.dtype == np.float16:
            n = n.view(np.uint16)
        if n.dtype != np.uint16:
            raise ValueError("grouped formats take binary16 scales")
        return np.ascontiguousarray(n)
    return _np(a, np.float32)


def decode(q, k_pool, v_pool, fmt: str, sel, cu, softmax_scale: float,
           k_scale=None, v_scale=None, rows=None, threads: int = 0) -> np.ndarray:
    """Oracle decode. Returns float64 [len(rows) or bs, Hq, D].

    q: bf16 [bs, Hq, D] (torch bf16 tensor or uint16 bits); k_pool/v_pool:
    [num_slots, Hkv, D] (bf16 bits / uint8 e4m3 / int8) or [num_slots, Hkv, D/2]
    uint8 (4-bit formats); sel int32 [n_sel]; cu int32 [bs+1]; scales float32
    (fp8 [1], int8/int4 [num_slots, Hkv]) or binary16 [num_slots, Hkv, D/group]
    for the grouped formats.
    """
    lib = _load()
    f = FORMATS[fmt]
    qn = _np(q)
    if qn.dtype != np.uint16:
        raise ValueError("q must be bf16")
    bs, Hq, D = qn.shape
    kn, vn = _np(k_pool), _np(v_pool)
    num_slots, Hkv = kn.shape[0], kn.shape[1]
    if fmt in NIBBLE:
        if kn.shape[2] * 2 != D:
            raise ValueError("4-bit pool rows must hold D/2 bytes")
    elif kn.shape[2] != D:
        raise ValueError("pool rows must hold D elements")
    sn = _np(sel, np.int32)
    cn = _np(cu, np.int32)
    if cn.shape[0] != bs + 1:
        raise ValueError("cu_seqlens must have bs+1 entries")
    ks, vs = _scales(k_scale, fmt), _scales(v_scale, fmt)
    if f != 0 and (ks is None or vs is None):
        raise ValueError("quantised pools need k_scale and v_scale")
    rn = _np(rows, np.int32) if rows is not None else None
    n_rows = bs if rn is None else rn.shape[0]
    out = np.zeros((n_rows, Hq, D), dtype=np.float64)
    rc = lib.orc_decode(_ptr(qn), Hq * D, D, _ptr(kn), _ptr(vn), f, num_slots, Hkv, D,
                        _ptr(ks), _ptr(vs), float(softmax_scale), _ptr(sn), sn.shape[0],
                        _ptr(cn), bs, Hq, _ptr(rn), n_rows, _ptr(out), int(threads))
    if rc != 0:
        raise OracleRefused({-1: "bad geometry", -2: "bad cu_seqlens",
                             -3: "slot id out of range"}.get(rc, str(rc)))
    return out


def decode_tiered(q, k_pool, v_pool, sel, cu, softmax_scale: float, k_scale, v_scale,
                  k_ring, v_ring, k_ring_scale, v_ring_scale, owner, rows=None,
                  threads: int = 0) -> np.ndarray:
    """Oracle decode over a tiered int8ring_int4 pool. Returns float64 [rows, Hq, D].

    k_pool/v_pool: int4_g32 rows [num_slots, Hkv, D/2] uint8 with binary16 scales
    [num_slots, Hkv, D/32]; k_ring/v_ring: int8_g64 rows [R, Hkv, D] with binary16
    scales [R, Hkv, D/64]; owner: int32 [R] (R a power of two; -1 = no owner)."""
    lib = _load()
    qn = _np(q)
    bs, Hq, D = qn.shape
    kn, vn = _np(k_pool), _np(v_pool)
    num_slots, Hkv = kn.shape[0], kn.shape[1]
    kr, vr = _np(k_ring).view(np.int8), _np(v_ring).view(np.int8)
    on = _np(owner, np.int32)
    R = on.shape[0]
    if kr.shape != (R, Hkv, D) or kn.shape[2] * 2 != D:
        raise ValueError("ring rows must be [R, Hkv, D] int8 and pool rows [slots, Hkv, D/2]")
    sn, cn = _np(sel, np.int32), _np(cu, np.int32)
    rn = _np(rows, np.int32) if rows is not None else None
    n_rows = bs if rn is None else rn.shape[0]
    out = np.zeros((n_rows, Hq, D), dtype=np.float64)
    ks, vs = _scales(k_scale, "int4_g32"), _scales(v_scale, "int4_g32")
    krs, vrs = _scales(k_ring_scale, "int8_g64"), _scales(v_ring_scale, "int8_g64")
    rc = lib.orc_decode_tiered(_ptr(qn), Hq * D, D, _ptr(kn), _ptr(vn), num_slots, Hkv, D,
                               _ptr(ks), _ptr(vs), _ptr(kr), _ptr(vr), _ptr(krs), _ptr(vrs),
                               _ptr(on), R, float(softmax_scale), _ptr(sn), sn.shape[0], _ptr(cn),
                               bs, Hq, _ptr(rn), n_rows, _ptr(out), int(threads))
    if rc != 0:
        raise OracleRefused({-1: "bad geometry", -2: "bad cu_seqlens",
                             -3: "slot id out of range"}.get(rc, str(rc)))
    return out


def write_tiered(x_k, x_v, slots, pools: dict) -> None:
    """The tiered write, in token order (a later token of the same write takes a
    ring row over an earlier one): for token i with slot s and ring position
    p = s & (R - 1), every head g gets the int4_g32 row (s, g) and the int8_g64
    ring row (p, g), and owner[p] = s. `pools` holds numpy arrays, updated in
    place: k_pool, v_pool (uint8 [slots, Hkv, D/2]), k_scale, v_scale (float16
    [slots, Hkv, D/32]), k_ring, v_ring (int8 [R, Hkv, D]), k_ring_scale,
    v_ring_scale (float16 [R, Hkv, D/64]), owner (int32 [R])."""
    xk, xv = _np(x_k), _np(x_v)
    n, Hkv, D = xk.shape
    sl = _np(slots, np.int32)
    R = pools["owner"].shape[0]
    for x, pool, sc, ring, rsc in ((xk, "k_pool", "k_scale", "k_ring", "k_ring_scale"),
                                   (xv, "v_pool", "v_scale", "v_ring", "v_ring_scale")):
        c4, s4 = quantize_rows(x.reshape(n * Hkv, D), "int4_g32")
        c8, s8 = quantize_rows(x.reshape(n * Hkv, D), "int8_g64")
        c4, s4 = c4.reshape(n, Hkv, -1), s4.reshape(n, Hkv, -1)
        c8, s8 = c8.reshape(n, Hkv, -1), s8.reshape(n, Hkv, -1)
        for i in range(n):
            s, pos = int(sl[i]), int(sl[i]) & (R - 1)
            pools[pool][s] = c4[i]
            pools[sc][s] = s4[i]
            pools[ring][pos] = c8[i]
            pools[rsc][pos] = s8[i]
    for i in range(n):
        pools["owner"][int(sl[i]) & (R - 1)] = sl[i]


def dequant_rows(pool, fmt: str, slots, g: int, scale=None) -> np.ndarray:
    """Exact FP64 dequantisation of pool rows (slot, g) for each slot in `slots`."""
    lib = _load()
    pn = _np(pool)
    Hkv = pn.shape[1]
    D = pn.shape[2] * (2 if fmt in NIBBLE else 1)
    sc = _scales(scale, fmt)
    out = np.zeros((len(slots), D), dtype=np.float64)
    for i, s in enumerate(slots):
        row = out[i]
        lib.orc_dequant_row(_ptr(pn), FORMATS[fmt], Hkv, D, _ptr(sc), int(s), int(g),
                            row.ctypes.data_as(ctypes.c_void_p))
    return out


def e4m3fn_to_double(byte: int) -> float:
    return _load().orc_e4m3fn_to_double(int(byte))


def int4_value(byte: int, hi: int) -> int:
    return _load().orc_int4_value(int(byte), int(hi))


def int4_offset_value(byte: int, hi: int) -> int:
    return _load().orc_int4_offset_value(int(byte), int(hi))


def fp16_to_double(bits: int) -> float:
    return _load().orc_fp16_to_double(int(bits))


def round_fp16_bits(v: float) -> int:
    """binary16 bits of a binary32 value rounded to nearest, ties to even."""
    return _load().orc_round_fp16(float(v))


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round every element of a float64 array to bf16 (ties to even); returns uint16 bits."""
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float64).ravel()
    bits = np.empty(flat.size, dtype=np.uint16)
    lib.orc_round_bf16_array(_ptr(flat), _ptr(bits), flat.size)
    return bits.reshape(np.shape(x))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 values of round_bf16_bits(x)."""
    bits = round_bf16_bits(x).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def e4m3fn_encode(v: float) -> int:
    """e4m3fn code of a binary32 value (nearest-even, saturating at +-448)."""
    return _load().orc_e4m3fn_encode(float(v))


def quantize_rows(x, fmt: str, fp8_scale: float = 1.0):
    """Quantise bf16 rows [n, D] as the KV write path does.

    Returns (codes, scales): codes uint8 [n, D] (bf16: uint16 bits [n, D];
    int8 / int8_g64: int8 [n, D]; int4 / int4_g32: uint8 [n, D/2]); scales
    float32 [n] for int8/int4, float16 [n, D/group] for the grouped formats,
    else None."""
    lib = _load()
    xn = _np(x)
    if xn.dtype != np.uint16 or xn.ndim != 2:
        raise ValueError("x must be bf16 [n, D]")
    n, D = xn.shape
    f = FORMATS[fmt]
    if fmt == "bf16":
        codes = np.empty((n, D), dtype=np.uint16)
    elif fmt in NIBBLE:
        codes = np.zeros((n, D // 2), dtype=np.uint8)
    else:
        codes = np.empty((n, D), dtype=np.uint8)
    if fmt in GROUP:
        scales = np.zeros((n, D // GROUP[fmt]), dtype=np.uint16)
    elif fmt in ("int8", "int4"):
        scales = np.zeros(n, dtype=np.float32)
    else:
        scales = None
    rc = lib.orc_quantize_rows(_ptr(xn), n, D, f, float(fp8_scale), _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("bad format or shape")
    if fmt in ("int8", "int8_g64"):
        codes = codes.view(np.int8)
    if fmt in GROUP:
        scales = scales.view(np.float16)
    return codes, scales


def max_threads() -> int:
    return _load().orc_max_threads()


# The step that produces the selected slots (exact top-k over compressed-block
# scores and index expansion) lives in topk.py: index work, plain numpy.
from .topk import TopkRefused, row_width, topk_blocks, topk_expand  # noqa: E402,F401
