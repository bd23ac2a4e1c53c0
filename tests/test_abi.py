"""The C ABI without a GPU: the library loads, exports every declared
symbol, the binding's structs match the header, and contract violations are
rejected on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from sparse_attention_paged_qsa_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = B.load()
    names = declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(lib, name), f"{name} declared in qsa.h but not exported"
    assert sorted(B.EXPORTED) == names
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    for name in names:
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_shipped_library_reads_no_environment_and_has_no_test_hook():
    lib = B.load()
    assert not hasattr(lib, "qsa_test_set_stall_stage")
    out = subprocess.run(["nm", "-D", "--undefined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    assert not re.search(r"\bgetenv\b", out), "libqsa.so imports getenv"
    # the test build carries the hook (and only the decode)
    test_lib = B.open_library(os.path.join(os.path.dirname(B.LIB_PATH), "libqsa_testhooks.so"))
    assert hasattr(test_lib, "qsa_test_set_stall_stage") and hasattr(test_lib, "qsa_decode")


def test_struct_layouts_match_header(tmp_path):
    src = tmp_path / "sizes.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "qsa.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(qsa_tensor),"
        " sizeof(qsa_kv_quant_meta), offsetof(qsa_kv_quant_meta, softmax_scale),"
        " offsetof(qsa_kv_quant_meta, max_ctas), sizeof(qsa_scratch_layout),"
        " offsetof(qsa_tensor, stride));return 0;}\n")
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()))
    assert got == [ctypes.sizeof(B.QsaTensor), ctypes.sizeof(B.QsaKvQuantMeta),
                   B.QsaKvQuantMeta.softmax_scale.offset, B.QsaKvQuantMeta.max_ctas.offset,
                   ctypes.sizeof(B.QsaScratchLayout), B.QsaTensor.stride.offset]


def test_version_and_strerror():
    lib = B.load()
    assert lib.qsa_version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.qsa_strerror(code)
    assert lib.qsa_strerror(-99) == b"unknown error"


def _host_call(q_shape=(2, 24, 256), pool_shape=(64, 2, 256), fmt="bf16", pool_dtype=None,
               capacity=100, q_offset=0, scales=False, scratch=True, cu_len=None, scale_offset=0):
    """Describe host tensors (never dereferenced) and call qsa_decode."""
    pd = pool_dtype or {"bf16": torch.bfloat16, "fp8_e4m3": torch.uint8, "int8": torch.int8,
                        "int4": torch.uint8, "int8_g64": torch.int8, "int4_g32": torch.uint8}[fmt]
    qbuf = torch.zeros(int(torch.tensor(q_shape).prod()) + 64, dtype=torch.bfloat16)
    q = qbuf[q_offset:q_offset + int(torch.tensor(q_shape).prod())].view(q_shape)
    k = torch.zeros(pool_shape, dtype=pd)
    v = torch.zeros(pool_shape, dtype=pd)
    bs = q_shape[0]
    sel = torch.zeros(10, dtype=torch.int32)
    cu = torch.zeros(cu_len or (bs + 1), dtype=torch.int32)
    out = torch.zeros(q_shape, dtype=torch.bfloat16)
    sc = torch.ones(pool_shape[0] * pool_shape[1] * 8 + 64, dtype=torch.float16)
    sc = sc[(-sc.data_ptr() // 2) % 8 + scale_offset:]   # 16-byte aligned, then offset
    meta = B.KVQuantMeta(fmt, capacity, sc if scales else None, sc if scales else None, 1 / 16)
    scr = torch.zeros(1 << 16, dtype=torch.uint8)
    lib = B.load()
    d = [B.describe(t) for t in (q, k, v)]
    m = meta.to_c()
    sd, cd, od = B.describe(sel), B.describe(cu), B.describe(out)
    base = scr.data_ptr()
    aligned = (base + 255) // 256 * 256
    rc = lib.qsa_decode(ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[2]),
                        ctypes.byref(m), ctypes.byref(sd), ctypes.byref(cd), ctypes.byref(od),
                        aligned if scratch else None, 1 << 15, None)
    return rc, lib.qsa_last_error_message().decode()


@pytest.mark.parametrize("kw, code, text", [
    (dict(q_shape=(0, 24, 256)), B.ERR_UNSUPPORTED, "batch size"),
    (dict(q_shape=(129, 24, 256)), B.ERR_UNSUPPORTED, "batch size"),
    (dict(q_shape=(2, 16, 256)), B.ERR_UNSUPPORTED, "query heads"),
    (dict(q_shape=(2, 24, 128)), B.ERR_UNSUPPORTED, "D = 256"),
    (dict(capacity=2056), B.ERR_UNSUPPORTED, "capacity"),
    (dict(capacity=0), B.ERR_UNSUPPORTED, "capacity"),
    (dict(pool_dtype=torch.float32), B.ERR_INVALID_ARGUMENT, "dtype"),
    (dict(pool_shape=(64, 1, 256)), B.ERR_INVALID_ARGUMENT, "Hkv=2"),
    (dict(fmt="int4", pool_shape=(64, 2, 256)), B.ERR_INVALID_ARGUMENT, "128"),
    (dict(fmt="int8"), B.ERR_INVALID_ARGUMENT, "scale"),
    (dict(fmt="int8_g64", pool_dtype=torch.uint8, scales=True), B.ERR_INVALID_ARGUMENT, "dtype"),
    (dict(fmt="int4_g32", pool_shape=(64, 2, 256), scales=True), B.ERR_INVALID_ARGUMENT, "128"),
    (dict(fmt="int4_g32", pool_shape=(64, 2, 128)), B.ERR_INVALID_ARGUMENT, "scale"),
    (dict(fmt="int8_g64", scales=True, scale_offset=2), B.ERR_MISALIGNED, "8-byte"),
    (dict(fmt="int4_g32", pool_shape=(64, 2, 128), scales=True, scale_offset=4), B.ERR_MISALIGNED,
     "16-byte"),
    (dict(q_offset=1), B.ERR_MISALIGNED, "aligned"),
    (dict(scratch=False), B.ERR_INVALID_ARGUMENT, "scratch"),
    (dict(cu_len=2), B.ERR_INVALID_ARGUMENT, "cu_seqlens"),
])
def test_contract_rejections_on_host(kw, code, text):
    rc, msg = _host_call(**kw)
    assert rc == code, msg
    assert text in msg


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        B.load()


def test_oracle_and_product_share_no_code():
    pkg = os.path.join(ROOT, "sparse_attention_paged_qsa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "qsa_oracle" not in text and "liboracle" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "sparse_attention_paged_qsa_gb300" not in text, f
            assert "qsa.h" not in text, f


def test_kv_write_rejections_on_host():
    lib = B.load()
    x = torch.zeros(4, 2, 256, dtype=torch.bfloat16)
    slots = torch.zeros(4, dtype=torch.int32)
    pool = torch.zeros(16, 2, 256, dtype=torch.int8)
    sc = torch.zeros(32)
    d = lambda t: ctypes.byref(B.describe(t))
    rc = lib.qsa_kv_write(2, d(x), d(x), d(slots), d(pool), d(pool), None, None, None, None)
    assert rc == B.ERR_INVALID_ARGUMENT and b"scale" in lib.qsa_last_error_message()
    rc = lib.qsa_kv_write(1, d(x), d(x), d(slots), d(pool), d(pool), sc.data_ptr(), sc.data_ptr(),
                          None, None)
    assert rc == B.ERR_INVALID_ARGUMENT and b"dtype" in lib.qsa_last_error_message()
    x3 = torch.zeros(4, 3, 256, dtype=torch.bfloat16)
    rc = lib.qsa_kv_write(2, d(x3), d(x3), d(slots), d(pool), d(pool), sc.data_ptr(), sc.data_ptr(),
                          None, None)
    assert rc == B.ERR_UNSUPPORTED
    # grouped pools: binary16 scales, 8- (int8_g64) / 16-byte (int4_g32) aligned
    h = torch.zeros(16 * 2 * 8 + 16, dtype=torch.float16)
    h = h[(-h.data_ptr() // 2) % 8:]
    rc = lib.qsa_kv_write(4, d(x), d(x), d(slots), d(pool), d(pool), h.data_ptr() + 4,
                          h.data_ptr(), None, None)
    assert rc == B.ERR_MISALIGNED and b"8-byte" in lib.qsa_last_error_message()
    pool4 = torch.zeros(16, 2, 128, dtype=torch.uint8)
    rc = lib.qsa_kv_write(5, d(x), d(x), d(slots), d(pool4), d(pool4), h.data_ptr() + 8,
                          h.data_ptr(), None, None)
    assert rc == B.ERR_MISALIGNED and b"16-byte" in lib.qsa_last_error_message()
    rc = lib.qsa_kv_write(5, d(x), d(x), d(slots), d(pool), d(pool), h.data_ptr(), h.data_ptr(),
                          None, None)
    assert rc == B.ERR_INVALID_ARGUMENT and b"dtype" in lib.qsa_last_error_message()
    empty = torch.zeros(0, 2, 256, dtype=torch.bfloat16)
    rc = lib.qsa_kv_write(2, d(empty), d(empty), d(torch.zeros(0, dtype=torch.int32)), d(pool),
                          d(pool), sc.data_ptr(), sc.data_ptr(), None, None)
    assert rc == B.OK  # nothing to write, nothing enqueued


def test_binding_rejects_host_tensors():
    """The C ABI takes device pointers; the binding refuses host tensors before the call."""
    q = torch.zeros(2, 24, 256, dtype=torch.bfloat16)
    pool = torch.zeros(8, 2, 256, dtype=torch.bfloat16)
    meta = B.KVQuantMeta("bf16", 4)
    with pytest.raises(B.QsaError, match="on the GPU"):
        B.qsa_decode(q, pool, pool, meta, torch.zeros(4, dtype=torch.int32),
                     torch.zeros(3, dtype=torch.int32), q, torch.zeros(1024, dtype=torch.uint8))
    with pytest.raises(B.QsaError, match="on the GPU"):
        B.qsa_kv_write("bf16", pool, pool, torch.zeros(8, dtype=torch.int32), pool, pool)


def _tier_call(ring_slots=64, drop=None, misalign=None, with_tier=True):
    """qsa_decode on a tiered pool with host tensors (never dereferenced)."""
    lib = B.load()
    q = torch.zeros(2, 24, 256, dtype=torch.bfloat16)
    pool = torch.zeros(64, 2, 128, dtype=torch.uint8)
    sc = torch.ones(64 * 2 * 8 + 64, dtype=torch.float16)
    sc = sc[(-sc.data_ptr() // 2) % 8:]
    ring = torch.zeros(ring_slots * 2 * 256 + 64, dtype=torch.int8)
    ring = ring[(-ring.data_ptr()) % 16:]
    rsc = torch.ones(ring_slots * 2 * 4 + 8, dtype=torch.float16)
    rsc = rsc[(-rsc.data_ptr() // 2) % 4:]
    owner = torch.full((max(ring_slots, 1),), -1, dtype=torch.int32)
    tier = {"k_ring": ring, "v_ring": ring, "k_ring_scale": rsc, "v_ring_scale": rsc, "owner": owner}
    t = B.tier_struct(tier)
    t.ring_slots = ring_slots
    if drop:
        setattr(t, drop, None)
    if misalign:
        setattr(t, misalign, getattr(t, misalign) + 2)
    m = B.KVQuantMeta("int8ring_int4", 100, sc, sc, 1 / 16).to_c()
    if with_tier:
        m.tier = ctypes.pointer(t)
    d = [B.describe(x) for x in (q, pool, pool)]
    sel, cu, out = torch.zeros(10, dtype=torch.int32), torch.zeros(3, dtype=torch.int32), q.clone()
    scr = torch.zeros(1 << 16, dtype=torch.uint8)
    aligned = (scr.data_ptr() + 255) // 256 * 256
    rc = lib.qsa_decode(ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[2]), ctypes.byref(m),
                        ctypes.byref(B.describe(sel)), ctypes.byref(B.describe(cu)),
                        ctypes.byref(B.describe(out)), aligned, 1 << 15, None)
    return rc, lib.qsa_last_error_message().decode()


@pytest.mark.parametrize("kw, code, text", [
    (dict(with_tier=False), B.ERR_INVALID_ARGUMENT, "tier"),
    (dict(ring_slots=48), B.ERR_INVALID_ARGUMENT, "power of two"),
    (dict(ring_slots=0), B.ERR_INVALID_ARGUMENT, "power of two"),
    (dict(drop="owner"), B.ERR_INVALID_ARGUMENT, "NULL"),
    (dict(misalign="k_ring"), B.ERR_MISALIGNED, "16-byte"),
    (dict(misalign="v_ring_scale"), B.ERR_MISALIGNED, "8-byte"),
])
def test_tiered_decode_rejections_on_host(kw, code, text):
    rc, msg = _tier_call(**kw)
    assert rc == code, msg
    assert text in msg


def _topk_host_call(bs=2, cap=4096, ratio=4, topk=2048, page=0, pt_cols=None, score_cols=None,
                    sel_len=None, cu_len=None, score_dtype=torch.float32, ctx_len=None):
    """Describe host tensors (never dereferenced) and call qsa_topk_expand."""
    scores = torch.zeros(bs, score_cols or cap // max(ratio, 1), dtype=score_dtype)
    ctx = torch.zeros(ctx_len or bs, dtype=torch.int32)
    pt = torch.zeros(bs, pt_cols or max(1, -(-cap // max(page, 1))), dtype=torch.int32)
    sel = torch.zeros(sel_len or bs * (topk + ratio - 1), dtype=torch.int32)
    cu = torch.zeros(cu_len or bs + 1, dtype=torch.int32)
    lib = B.load()
    prm = B.QsaTopkParams(topk, ratio, cap, page)
    d = [B.describe(t) for t in (scores, ctx, pt if page else None, sel, cu)]
    rc = lib.qsa_topk_expand(ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[2]),
                             ctypes.byref(prm), ctypes.byref(d[3]), ctypes.byref(d[4]), None, None)
    return rc, lib.qsa_last_error_message().decode()


@pytest.mark.parametrize("kw, code, text", [
    (dict(ratio=0), B.ERR_UNSUPPORTED, "compress ratio"),
    (dict(ratio=65, topk=65 * 4), B.ERR_UNSUPPORTED, "compress ratio"),
    (dict(topk=2046), B.ERR_UNSUPPORTED, "multiple"),
    (dict(topk=2056, ratio=8), B.ERR_UNSUPPORTED, "2055"),
    (dict(cap=262145), B.ERR_UNSUPPORTED, "capacity"),
    (dict(bs=129), B.ERR_UNSUPPORTED, "bs"),
    (dict(score_cols=1000), B.ERR_INVALID_ARGUMENT, "scores"),
    (dict(score_dtype=torch.bfloat16), B.ERR_INVALID_ARGUMENT, "scores"),
    (dict(page=48), B.ERR_UNSUPPORTED, "page size"),
    (dict(page=64, pt_cols=63), B.ERR_INVALID_ARGUMENT, "page_table"),
    (dict(sel_len=2 * 2051 - 1), B.ERR_INVALID_ARGUMENT, "sel_indices"),
    (dict(cu_len=2), B.ERR_INVALID_ARGUMENT, "cu_seqlens"),
])
def test_topk_rejections_on_host(kw, code, text):
    rc, msg = _topk_host_call(**kw)
    assert rc == code, msg
    assert text in msg


def test_topk_struct_layout_matches_header(tmp_path):
    src = tmp_path / "tk.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "qsa.h"\n'
                   'int main(void){printf("%zu %zu\\n", sizeof(qsa_topk_params),'
                   ' offsetof(qsa_topk_params, page_size));return 0;}\n')
    exe = tmp_path / "tk"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()))
    assert got == [ctypes.sizeof(B.QsaTopkParams), B.QsaTopkParams.page_size.offset]
