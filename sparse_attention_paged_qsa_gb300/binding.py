"""Thin ctypes binding over libqsa (include/qsa.h).

Argument marshalling only: torch tensors are described by pointer, dtype,
shape and strides and handed to the C ABI; every step of the decode runs in
the library's CUDA kernel. There is no fallback path: if libqsa.so is missing
the first call raises.
"""
from __future__ import annotations

import ctypes
import struct
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqsa.so")

# include/qsa.h enums
DTYPE_BF16, DTYPE_UINT8, DTYPE_INT8, DTYPE_INT32, DTYPE_FLOAT32 = 1, 2, 3, 4, 5
KV_FORMATS = {"bf16": 0, "fp8_e4m3": 1, "int8": 2, "int4": 3, "int8_g64": 4, "int4_g32": 5,
              "int8ring_int4": 6}
OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_SCRATCH_TOO_SMALL, ERR_MISALIGNED, ERR_CUDA = (
    0, -1, -2, -3, -4, -5)
DEVERR_SLOT_RANGE, DEVERR_CU_SEQLENS, DEVERR_TIMEOUT, DEVERR_CTX_LEN = 1, 2, 4, 8

_TORCH_DTYPES = {
    torch.bfloat16: DTYPE_BF16,
    torch.uint8: DTYPE_UINT8,
    torch.int8: DTYPE_INT8,
    torch.int32: DTYPE_INT32,
    torch.float32: DTYPE_FLOAT32,
}

EXPORTED = (
    "qsa_decode", "qsa_decode_scratch_bytes", "qsa_decode_grid", "qsa_decode_scratch_layout",
    "qsa_scratch_init", "qsa_scratch_error", "qsa_strerror", "qsa_last_error_message",
    "qsa_version", "qsa_decode_static_scratch", "qsa_kv_write", "qsa_kv_write_tiered",
    "qsa_topk_expand",
)


class QsaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class QsaKvTier(ctypes.Structure):
    _fields_ = [("k_ring", ctypes.c_void_p), ("v_ring", ctypes.c_void_p),
                ("k_ring_scale", ctypes.c_void_p), ("v_ring_scale", ctypes.c_void_p),
                ("owner", ctypes.c_void_p), ("ring_slots", ctypes.c_int32)]


class QsaKvQuantMeta(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("softmax_scale", ctypes.c_float), ("max_ctas", ctypes.c_int32),
                ("tier", ctypes.POINTER(QsaKvTier))]


def tier_struct(tier: dict) -> QsaKvTier:
    """qsa_kv_tier from a dict of device tensors (k_ring, v_ring, k_ring_scale,
    v_ring_scale, owner); the ring size is owner's length."""
    t = QsaKvTier()
    for key in ("k_ring", "v_ring", "k_ring_scale", "v_ring_scale", "owner"):
        setattr(t, key, tier[key].data_ptr())
    t.ring_slots = int(tier["owner"].numel())
    return t


class QsaTopkParams(ctypes.Structure):
    _fields_ = [("token_topk", ctypes.c_int32), ("compress_ratio", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("page_size", ctypes.c_int32)]


class QsaScratchLayout(ctypes.Structure):
    _fields_ = [("error_word_offset", ctypes.c_size_t), ("counters_offset", ctypes.c_size_t),
                ("counters_count", ctypes.c_size_t), ("partials_offset", ctypes.c_size_t),
                ("partial_slot_bytes", ctypes.c_size_t), ("total_bytes", ctypes.c_size_t)]


class QsaError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{message} (code {code})")
        self.code = code


_lib = None


def load() -> ctypes.CDLL:
    """Load libqsa.so from the package directory (raises if it was not built)."""
    global _lib
    if _lib is None:
        _lib = open_library(LIB_PATH)
    return _lib


def _signatures():
    """(restype, argtypes) of every export of qsa.h."""
    P, T, M = ctypes.POINTER, ctypes.POINTER(QsaTensor), ctypes.POINTER(QsaKvQuantMeta)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    return {
        "qsa_decode": (ctypes.c_int, [T, T, T, M, T, T, T, vp, ctypes.c_size_t, vp]),
        "qsa_decode_static_scratch": (ctypes.c_int, [T, T, T, M, T, T, T, vp]),
        "qsa_kv_write": (ctypes.c_int, [i32, T, T, T, T, T, vp, vp, vp, vp]),
        "qsa_kv_write_tiered": (ctypes.c_int, [T, T, T, T, T, vp, vp, P(QsaKvTier), vp, vp]),
        "qsa_decode_scratch_bytes": (ctypes.c_size_t, [i32] * 3),
        "qsa_decode_grid": (i32, [i32] * 4),
        "qsa_decode_scratch_layout": (ctypes.c_int, [i32] * 3 + [P(QsaScratchLayout)]),
        "qsa_scratch_init": (ctypes.c_int, [vp, ctypes.c_size_t, vp]),
        "qsa_scratch_error": (ctypes.c_int, [vp, P(i32), i32, vp]),
        "qsa_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "qsa_last_error_message": (ctypes.c_char_p, []),
        "qsa_version": (ctypes.c_int, []),
        "qsa_topk_expand": (ctypes.c_int, [T, T, T, P(QsaTopkParams), T, T, vp, vp]),
    }


def open_library(path: str) -> ctypes.CDLL:
    """Open a build of the C ABI at `path` and declare the signatures of the
    qsa.h exports it has (a test build carries the decode only)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _signatures().items():
        if hasattr(lib, name):
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
    return lib


def _check(rc: int) -> None:
    if rc != OK:
        lib = load()
        msg = lib.qsa_last_error_message().decode() or lib.qsa_strerror(rc).decode()
        raise QsaError(rc, msg)


# qsa_tensor as packed bytes: void* data, int32 dtype, int32 ndim, int64 shape[4],
# int64 stride[4] (one pack is faster than filling the ctypes arrays field by field)
_TENSOR_PACK = struct.Struct("<qii4q4q")
_PAD = ((), (0,), (0, 0), (0, 0, 0), (0, 0, 0, 0))
assert _TENSOR_PACK.size == ctypes.sizeof(QsaTensor)


def describe(t: Optional[torch.Tensor]) -> QsaTensor:
    """qsa_tensor view of a torch tensor (no copy)."""
    if t is None:
        return QsaTensor()
    nd = t.dim()
    if nd > 4:
        raise ValueError("at most 4 dimensions")
    pad = _PAD[4 - nd]
    return QsaTensor.from_buffer_copy(_TENSOR_PACK.pack(
        t.data_ptr() if t.numel() else 0, _TORCH_DTYPES.get(t.dtype, 0), nd,
        *t.shape, *pad, *t.stride(), *pad))


@dataclass
class KVQuantMeta:
    """Python mirror of qsa_kv_quant_meta."""

    format: str = "bf16"
    capacity: int = 2055
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    softmax_scale: float = 1.0 / 16.0
    max_ctas: int = 0
    tier: Optional[dict] = None   # int8ring_int4: k_ring, v_ring, k_ring_scale, v_ring_scale, owner

    def to_c(self) -> QsaKvQuantMeta:
        m = QsaKvQuantMeta()
        if self.tier is not None:
            m._tier = tier_struct(self.tier)      # kept alive with the struct
            m.tier = ctypes.pointer(m._tier)
        m.format = KV_FORMATS[self.format]
        m.capacity = int(self.capacity)
        m.k_scale = self.k_scale.data_ptr() if self.k_scale is not None else None
        m.v_scale = self.v_scale.data_ptr() if self.v_scale is not None else None
        m.softmax_scale = float(self.softmax_scale)
        m.max_ctas = int(self.max_ctas)
        return m


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _require_device(*tensors) -> None:
    """The library takes device pointers; a host tensor here is a caller error."""
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise QsaError(ERR_INVALID_ARGUMENT, "every tensor must be on the GPU (got a host tensor)")


def qsa_decode(q, k_pool, v_pool, kv_quant_meta: KVQuantMeta, sel_indices, cu_seqlens, out,
               scratch, stream=None) -> None:
    """Enqueue one packed QSA decode (see include/qsa.h). Raises QsaError on a contract error."""
    _require_device(q, k_pool, v_pool, sel_indices, cu_seqlens, out, scratch,
                    kv_quant_meta.k_scale, kv_quant_meta.v_scale,
                    *((kv_quant_meta.tier or {}).values()))
    lib = load()
    meta = kv_quant_meta.to_c()
    args = [describe(t) for t in (q, k_pool, v_pool)]
    sel_d, cu_d, out_d = describe(sel_indices), describe(cu_seqlens), describe(out)
    rc = lib.qsa_decode(ctypes.byref(args[0]), ctypes.byref(args[1]), ctypes.byref(args[2]),
                        ctypes.byref(meta), ctypes.byref(sel_d), ctypes.byref(cu_d),
                        ctypes.byref(out_d), scratch.data_ptr() if scratch is not None else None,
                        scratch.numel() * scratch.element_size() if scratch is not None else 0,
                        _stream_handle(stream))
    _check(rc)


def qsa_kv_write(fmt: str, k_new, v_new, slots, k_pool, v_pool, k_scale=None, v_scale=None,
                 error_word=None, stream=None) -> None:
    """Enqueue one quantise + scatter write of new K/V rows (see include/qsa.h)."""
    _require_device(k_new, v_new, slots, k_pool, v_pool, k_scale, v_scale, error_word)
    lib = load()
    d = [describe(t) for t in (k_new, v_new, slots, k_pool, v_pool)]
    ptr = lambda t: t.data_ptr() if t is not None else None
    rc = lib.qsa_kv_write(KV_FORMATS[fmt], *(ctypes.byref(x) for x in d), ptr(k_scale),
                          ptr(v_scale), ptr(error_word), _stream_handle(stream))
    _check(rc)


def qsa_kv_write_tiered(k_new, v_new, slots, k_pool, v_pool, k_scale, v_scale, tier: dict,
                        error_word=None, stream=None) -> None:
    """Enqueue the two-kernel write of a tiered int8ring_int4 pool (see include/qsa.h)."""
    _require_device(k_new, v_new, slots, k_pool, v_pool, k_scale, v_scale, error_word,
                    *tier.values())
    lib = load()
    d = [describe(t) for t in (k_new, v_new, slots, k_pool, v_pool)]
    ts = tier_struct(tier)
    ptr = lambda t: t.data_ptr() if t is not None else None
    rc = lib.qsa_kv_write_tiered(*(ctypes.byref(x) for x in d), ptr(k_scale), ptr(v_scale),
                                 ctypes.byref(ts), ptr(error_word), _stream_handle(stream))
    _check(rc)


def qsa_topk_expand(scores, ctx_lens, sel_indices, cu_seqlens, token_topk: int = 2048,
                    compress_ratio: int = 4, capacity: int = 262144, page_table=None,
                    page_size: int = 0, error_word=None, stream=None) -> None:
    """Enqueue the exact top-k + index expansion that fills sel_indices and
    cu_seqlens for qsa_decode (see include/qsa.h). page_size > 0 needs page_table."""
    _require_device(scores, ctx_lens, sel_indices, cu_seqlens, page_table, error_word)
    lib = load()
    prm = QsaTopkParams(int(token_topk), int(compress_ratio), int(capacity), int(page_size))
    d = [describe(t) for t in (scores, ctx_lens, page_table, sel_indices, cu_seqlens)]
    rc = lib.qsa_topk_expand(*(ctypes.byref(x) for x in d[:3]), ctypes.byref(prm),
                             ctypes.byref(d[3]), ctypes.byref(d[4]),
                             error_word.data_ptr() if error_word is not None else None,
                             _stream_handle(stream))
    _check(rc)


def qsa_decode_scratch_bytes(bs: int, num_q_heads: int, capacity: int) -> int:
    n = load().qsa_decode_scratch_bytes(bs, num_q_heads, capacity)
    if n == 0:
        _check(ERR_UNSUPPORTED)
    return n


def qsa_decode_grid(bs: int, num_q_heads: int, capacity: int, max_ctas: int = 0) -> int:
    g = load().qsa_decode_grid(bs, num_q_heads, capacity, max_ctas)
    if g < 0:
        _check(g)
    return g


def qsa_decode_scratch_layout(bs: int, num_q_heads: int, capacity: int) -> dict:
    ly = QsaScratchLayout()
    _check(load().qsa_decode_scratch_layout(bs, num_q_heads, capacity, ctypes.byref(ly)))
    return {k: getattr(ly, k) for k, _ in QsaScratchLayout._fields_}


def qsa_scratch_init(scratch: torch.Tensor, stream=None) -> None:
    _check(load().qsa_scratch_init(scratch.data_ptr(), scratch.numel() * scratch.element_size(),
                                   _stream_handle(stream)))


def qsa_scratch_error(scratch: torch.Tensor, clear: bool = False, stream=None) -> int:
    flags = ctypes.c_int32(0)
    _check(load().qsa_scratch_error(scratch.data_ptr(), ctypes.byref(flags), int(clear),
                                    _stream_handle(stream)))
    return flags.value


def alloc_scratch(bs: int, num_q_heads: int, capacity: int, device=None) -> torch.Tensor:
    """Allocate (torch caching allocator) and zero a scratch buffer for these sizes."""
    n = qsa_decode_scratch_bytes(bs, num_q_heads, capacity)
    buf = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    qsa_scratch_init(buf)
    return buf


def version() -> int:
    return load().qsa_version()
