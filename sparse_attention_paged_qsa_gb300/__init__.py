"""Packed Qwen-sparse-attention (QSA) decode for NVIDIA GB300 (sm_103a).

The compute lives in libqsa.so (CUDA kernels behind the C ABI declared in
include/qsa.h: the decode, the quantising KV write, and the exact top-k + index
expansion that produces the decode's selected slots); ``binding`` marshals torch tensors into that ABI, and
``inputs`` generates seeded synthetic workloads.
"""
from .binding import (  # noqa: F401
    KVQuantMeta,
    QsaError,
    alloc_scratch,
    qsa_decode,
    qsa_decode_grid,
    qsa_decode_scratch_bytes,
    qsa_decode_scratch_layout,
    qsa_kv_write,
    qsa_kv_write_tiered,
    qsa_scratch_error,
    qsa_scratch_init,
    qsa_topk_expand,
    version,
)

__all__ = [
    "KVQuantMeta", "QsaError", "alloc_scratch", "qsa_decode", "qsa_decode_grid",
    "qsa_decode_scratch_bytes", "qsa_decode_scratch_layout", "qsa_kv_write", "qsa_kv_write_tiered", "qsa_scratch_error",
    "qsa_scratch_init", "qsa_topk_expand", "version",
]
