"""The C-ABI library loads, exports every symbol include/pagedkv.h declares,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

from paged_attention_kv_gb300 import binding as pkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedkv.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))


def test_header_declarations_are_exported():
    names = _declared()
    assert {"paged_slot_mapping", "paged_kv_write", "paged_attention"} <= names
    lib = ctypes.CDLL(pkv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(pkv.EXPORTED)


def test_codes_match_header():
    text = open(HEADER).read()
    for name, val in re.findall(r"#define (PKV_(?:E_\w+|OK|DEV_\w+))\s+\(?(-?(?:0x)?[0-9a-fA-F]+)\)?", text):
        assert getattr(pkv, name) == int(val, 0), name
    for code in range(-9, 1):
        assert pkv.status_string(code) != "unknown status code"


def test_pool_bytes_follow_block_formula():
    # page 2 block-size note: 2 * 16 * Hkv * D * 2 bytes per block
    assert pkv.pkv_kv_cache_bytes(1, 4, 64) == 16384
    assert pkv.pkv_kv_cache_bytes(1, 8, 128) == 65536
    assert pkv.pkv_kv_cache_bytes(46000, 8, 128) == 46000 * 65536


def _desc(nb=64, bs=16, hkv=4, d=64):
    return pkv.CacheDesc(nb, bs, hkv, d)


def _attn(desc, q=0x1000, t=2, hq=32, kv=0x2000, bt=0x3000, r=2, mbr=3, sl=0x4000, qsl=0x5000, out=0x6000,
          ws=0x7000, wsb=1 << 30):
    vp = ctypes.c_void_p
    return pkv.LIB.paged_attention(vp(q), t, hq, vp(kv), ctypes.byref(desc), vp(bt), r, mbr, vp(sl), vp(qsl),
                                   ctypes.c_float(0.125), vp(out), vp(ws), wsb, vp(0))


def test_attention_host_validation():
    # None of these reaches the GPU: the call returns before any CUDA API use.
    assert _attn(_desc(bs=8)) == pkv.PKV_E_BLOCK_SIZE
    assert _attn(_desc(d=96)) == pkv.PKV_E_HEAD_SIZE
    assert _attn(_desc(hkv=5)) == pkv.PKV_E_GQA
    assert _attn(_desc(), hq=0) == pkv.PKV_E_GQA
    assert _attn(_desc(), q=0) == pkv.PKV_E_NULL
    assert _attn(_desc(), out=0) == pkv.PKV_E_NULL
    assert _attn(_desc(), q=0x1008) == pkv.PKV_E_ALIGN
    assert _attn(_desc(), ws=0x7010) == pkv.PKV_E_ALIGN
    assert _attn(_desc(), t=-1) == pkv.PKV_E_DIMS
    assert _attn(_desc(nb=0)) == pkv.PKV_E_DIMS
    assert _attn(_desc(), wsb=16) == pkv.PKV_E_WORKSPACE
    assert _attn(_desc(), t=0) == pkv.PKV_OK          # empty batch: nothing to do
    assert pkv.LIB.paged_attention(None, 2, 32, None, None, None, 2, 3, None, None, ctypes.c_float(1.0), None,
                                   None, 0, None) == pkv.PKV_E_NULL


def test_kv_write_and_slot_host_validation():
    vp = ctypes.c_void_p
    lib = pkv.LIB
    assert lib.paged_kv_write(vp(0x1000), vp(0x2000), vp(0x3000), 4, vp(0x4000), ctypes.byref(_desc(bs=32)),
                              None, None) == pkv.PKV_E_BLOCK_SIZE
    assert lib.paged_kv_write(vp(0x1000), vp(0x2000), vp(0x3000), 4, vp(0x4000), ctypes.byref(_desc(d=36)),
                              None, None) == pkv.PKV_E_HEAD_SIZE
    assert lib.paged_kv_write(vp(0x1004), vp(0x2000), vp(0x3000), 4, vp(0x4000), ctypes.byref(_desc()),
                              None, None) == pkv.PKV_E_ALIGN
    assert lib.paged_kv_write(None, vp(0x2000), vp(0x3000), 4, vp(0x4000), ctypes.byref(_desc()),
                              None, None) == pkv.PKV_E_NULL
    assert lib.paged_kv_write(None, None, None, 0, None, ctypes.byref(_desc()), None, None) == pkv.PKV_OK
    assert lib.paged_slot_mapping(vp(0x1000), 2, 3, vp(0x2000), vp(0x3000), 4, 0, vp(0x4000), None,
                                  None) == pkv.PKV_E_DIMS
    assert lib.paged_slot_mapping(None, 2, 3, vp(0x2000), vp(0x3000), 4, 64, vp(0x4000), None,
                                  None) == pkv.PKV_E_NULL
    assert lib.paged_slot_mapping(vp(0x1002), 2, 3, vp(0x2000), vp(0x3000), 4, 64, vp(0x4000), None,
                                  None) == pkv.PKV_E_ALIGN
    assert lib.paged_slot_mapping(None, 0, 0, None, None, 0, 64, None, None, None) == pkv.PKV_OK


def test_read_status_rejects_null():
    v = ctypes.c_int32(0)
    assert pkv.LIB.pkv_read_status(None, None, ctypes.byref(v)) == pkv.PKV_E_NULL


def test_binding_rejects_wrong_tensors():
    import torch
    q = torch.zeros(2, 32, 64, dtype=torch.float32)
    with pytest.raises((TypeError, ValueError)):
        pkv.paged_attention(q, q, q, q, q, 0.1)


def test_min_workspace_is_host_only_and_below_default_layout():
    d = _desc(nb=1000, hkv=8, d=128)
    out = ctypes.c_size_t(0)
    assert pkv.LIB.paged_attention_min_workspace_bytes(256, 256, 32, ctypes.byref(d), ctypes.byref(out)) == 0
    assert out.value > 0
    # A workspace one byte short is rejected before any CUDA call.
    assert _attn(d, t=256, r=256, wsb=out.value - 1) == pkv.PKV_E_WORKSPACE


def _pipeline_desc(**kw):
    d = pkv.PipelineDesc()
    d.depth = 2
    for i in range(2):
        d.host_in[i], d.dev_in[i] = 0x100000 * (i + 1), 0x200000 * (i + 1)
        d.slot_mapping[i], d.out[i] = 0x300000 + 0x1000 * i, 0x400000 + 0x10000 * i
    T, hq, hkv, D, R, M = 4, 32, 8, 128, 4, 8
    d.off_q, d.off_k, d.off_v = 0, T * hq * D * 2, T * hq * D * 2 + T * hkv * D * 2
    d.off_block_table = d.off_v + T * hkv * D * 2
    d.off_seq_lens = d.off_block_table + R * M * 4
    d.off_query_start_loc = d.off_seq_lens + 256
    d.in_bytes = d.off_query_start_loc + 256
    d.num_tokens, d.num_q_heads, d.max_num_reqs, d.max_blocks_per_req = T, hq, R, M
    d.cache = _desc(nb=64, hkv=hkv, d=D)
    d.status, d.workspace, d.workspace_bytes, d.scale = 0x500000, 0x600000, 1 << 20, 0.088
    d.h2d_stream, d.compute_stream, d.d2h_stream = 0x11, 0x22, 0x33
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_pipeline_create_validates_the_description_before_any_cuda_call():
    h = ctypes.c_void_p(0)
    create = pkv.LIB.pkv_pipeline_create
    assert create(None, ctypes.byref(h)) == pkv.PKV_E_NULL
    assert create(ctypes.byref(_pipeline_desc(depth=0)), ctypes.byref(h)) == pkv.PKV_E_DIMS
    assert create(ctypes.byref(_pipeline_desc(depth=5)), ctypes.byref(h)) == pkv.PKV_E_DIMS
    assert create(ctypes.byref(_pipeline_desc(num_q_heads=12)), ctypes.byref(h)) == pkv.PKV_E_GQA
    assert create(ctypes.byref(_pipeline_desc(status=None)), ctypes.byref(h)) == pkv.PKV_E_NULL
    bad = _pipeline_desc()
    bad.in_bytes = bad.off_query_start_loc + 8          # query_start_loc does not fit
    assert create(ctypes.byref(bad), ctypes.byref(h)) == pkv.PKV_E_DIMS
    bad = _pipeline_desc()
    bad.off_k += 8                                      # k not 16-byte aligned
    assert create(ctypes.byref(bad), ctypes.byref(h)) == pkv.PKV_E_DIMS
    bad = _pipeline_desc()
    bad.cache = _desc(nb=64, hkv=8, d=96)               # attention head size
    assert create(ctypes.byref(bad), ctypes.byref(h)) == pkv.PKV_E_HEAD_SIZE
    assert h.value is None
    slot = ctypes.c_int32(0)
    assert pkv.LIB.pkv_pipeline_next(None, ctypes.byref(slot)) == pkv.PKV_E_NULL
    assert pkv.LIB.pkv_pipeline_submit(None, 1, None, None, -1) == pkv.PKV_E_NULL
    assert pkv.LIB.pkv_pipeline_sync(None) == pkv.PKV_E_NULL
    assert pkv.LIB.pkv_pipeline_destroy(None) == pkv.PKV_OK


def test_fused_kv_write_host_validation():
    vp = ctypes.c_void_p
    f = pkv.LIB.paged_kv_write_slots
    d = ctypes.byref(_desc())
    ok = dict(k=vp(0x1000), v=vp(0x2000), bt=vp(0x3000), sl=vp(0x4000), qsl=vp(0x5000), kv=vp(0x6000),
              slots=vp(0x7000))

    def call(r=2, mbr=3, t=4, desc=d, **kw):
        a = {**ok, **kw}
        return f(a["k"], a["v"], a["bt"], r, mbr, a["sl"], a["qsl"], t, a["kv"], desc, a["slots"], None, None)
    assert call(t=0) == pkv.PKV_OK
    assert call(k=None) == pkv.PKV_E_NULL
    assert call(slots=None) == pkv.PKV_E_NULL
    assert call(qsl=None) == pkv.PKV_E_NULL
    assert call(k=vp(0x1004)) == pkv.PKV_E_ALIGN
    assert call(bt=vp(0x3002)) == pkv.PKV_E_ALIGN
    assert call(r=0) == pkv.PKV_E_DIMS
    assert call(t=-1) == pkv.PKV_E_DIMS
    assert call(desc=ctypes.byref(_desc(bs=32))) == pkv.PKV_E_BLOCK_SIZE
