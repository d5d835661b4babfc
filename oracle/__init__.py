"""fp64 CPU oracle for paged-KV attention (ctypes wrapper over ``oracle.c``).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package. The product path never
does, and the oracle shares no code with it.

Every array crosses as numpy: bf16 tensors as ``uint16`` bit patterns, index
tables as ``int32``. What each function computes, and the passage of "Inside
vLLM: Anatomy of a High-Throughput LLM Inference System" it follows, is stated
in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")

_STATUS = {
    0: "ok",
    -1: "bad argument",
    -2: "query_start_loc is not a valid ragged offset array",
    -3: "a request has more new tokens than context, or more context than its block table holds",
    -4: "a block id is outside the pool",
    -5: "a slot is outside the pool",
    -6: "out of memory",
}

_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; run __graft_entry__.build() first")
        lib = ctypes.CDLL(LIB_PATH)
        i32p = ctypes.POINTER(ctypes.c_int32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.orc_block_bytes.restype = ctypes.c_int64
        lib.orc_block_bytes.argtypes = [ctypes.c_int] * 4
        lib.orc_blocks_needed.restype = ctypes.c_int64
        lib.orc_blocks_needed.argtypes = [ctypes.c_int64, ctypes.c_int]
        lib.orc_slot_mapping.restype = ctypes.c_int
        lib.orc_slot_mapping.argtypes = [i32p, ctypes.c_int, ctypes.c_int, i32p, i32p,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p]
        lib.orc_kv_write.restype = ctypes.c_int
        lib.orc_kv_write.argtypes = [u16p, u16p, i32p, ctypes.c_int, u16p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.orc_kv_gather_blocks.restype = ctypes.c_int
        lib.orc_kv_gather_blocks.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             i32p, ctypes.c_int, u16p]
        lib.orc_kv_scatter_blocks.restype = ctypes.c_int
        lib.orc_kv_scatter_blocks.argtypes = [u16p, i32p, ctypes.c_int, u16p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int]
        lib.orc_paged_attention_rows.restype = ctypes.c_int
        lib.orc_paged_attention_rows.argtypes = [
            u16p, ctypes.c_int, ctypes.c_int,
            u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            i32p, ctypes.c_int, ctypes.c_int, i32p, i32p, ctypes.c_double,
            i32p, i32p, ctypes.c_int64, f64p, ctypes.c_int]
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: {_STATUS.get(rc, rc)}")


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def block_bytes(block_size: int, num_kv_heads: int, head_size: int, dtype_bytes: int) -> int:
    """Bytes of one KV block of one layer (page 2, the block-size note)."""
    return int(_load().orc_block_bytes(block_size, num_kv_heads, head_size, dtype_bytes))


def blocks_needed(tokens: int, block_size: int = 16) -> int:
    """ceil(tokens / block_size) ("Scheduler", allocate_slots step 1)."""
    return int(_load().orc_blocks_needed(tokens, block_size))


def slot_mapping(block_table, seq_lens, query_start_loc, num_blocks: int, block_size: int = 16) -> np.ndarray:
    """int32 slot per new token of the flattened batch."""
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    num_reqs = sl.shape[0]
    num_tokens = int(qsl[-1]) if num_reqs else 0
    out = np.full(num_tokens, -1, dtype=np.int32)
    mbr = bt.shape[1] if bt.ndim == 2 else 0
    rc = _load().orc_slot_mapping(_ptr(bt, ctypes.c_int32), num_reqs, mbr, _ptr(sl, ctypes.c_int32),
                                  _ptr(qsl, ctypes.c_int32), num_tokens, block_size, num_blocks,
                                  _ptr(out, ctypes.c_int32))
    _check(rc, "slot_mapping")
    return out


def kv_write(kv_cache: np.ndarray, k, v, slots) -> None:
    """Scatter K/V rows into ``kv_cache`` (uint16 [NB][2][Hkv][B][D]) in place."""
    assert kv_cache.dtype == np.uint16 and kv_cache.flags.c_contiguous and kv_cache.ndim == 5
    nb, two, hkv, bs, d = kv_cache.shape
    assert two == 2
    k = _c(k, np.uint16).reshape(-1, hkv, d)
    v = _c(v, np.uint16).reshape(-1, hkv, d)
    s = _c(slots, np.int32)
    assert k.shape == v.shape and k.shape[0] == s.shape[0]
    rc = _load().orc_kv_write(_ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), _ptr(s, ctypes.c_int32),
                              s.shape[0], _ptr(kv_cache, ctypes.c_uint16), nb, bs, hkv, d)
    _check(rc, "kv_write")


def kv_gather_blocks(kv_cache: np.ndarray, block_ids) -> np.ndarray:
    """uint16 [n][2][Hkv][B][D]: copies of the pool blocks block_ids[i]."""
    assert kv_cache.dtype == np.uint16 and kv_cache.flags.c_contiguous and kv_cache.ndim == 5
    nb, _, hkv, bs, d = kv_cache.shape
    ids = _c(block_ids, np.int32)
    out = np.zeros((ids.shape[0], 2, hkv, bs, d), dtype=np.uint16)
    rc = _load().orc_kv_gather_blocks(_ptr(kv_cache, ctypes.c_uint16), nb, bs, hkv, d, _ptr(ids, ctypes.c_int32),
                                      ids.shape[0], _ptr(out, ctypes.c_uint16))
    _check(rc, "kv_gather_blocks")
    return out


def kv_scatter_blocks(staging, block_ids, kv_cache: np.ndarray) -> None:
    """Writes staging[i] into pool block block_ids[i] (in place)."""
    assert kv_cache.dtype == np.uint16 and kv_cache.flags.c_contiguous and kv_cache.ndim == 5
    nb, _, hkv, bs, d = kv_cache.shape
    ids = _c(block_ids, np.int32)
    st = _c(staging, np.uint16)
    assert st.size == ids.shape[0] * 2 * hkv * bs * d
    rc = _load().orc_kv_scatter_blocks(_ptr(st, ctypes.c_uint16), _ptr(ids, ctypes.c_int32), ids.shape[0],
                                       _ptr(kv_cache, ctypes.c_uint16), nb, bs, hkv, d)
    _check(rc, "kv_scatter_blocks")


def paged_attention(q, kv_cache: np.ndarray, block_table, seq_lens, query_start_loc, scale: float,
                    rows=None, num_threads: int | None = None) -> np.ndarray:
    """fp64 attention output.

    q: uint16 [T][Hq][D]. With ``rows=None`` returns [T][Hq][D]; otherwise
    ``rows`` is an int array [N][2] of (token, q head) pairs and the result is
    [N][D].
    """
    q = _c(q, np.uint16)
    t, hq, d = q.shape
    assert kv_cache.dtype == np.uint16 and kv_cache.flags.c_contiguous and kv_cache.ndim == 5
    nb, _, hkv, bs, d2 = kv_cache.shape
    assert d2 == d
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    if rows is None:
        tok = np.repeat(np.arange(t, dtype=np.int32), hq)
        head = np.tile(np.arange(hq, dtype=np.int32), t)
    else:
        rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
        tok = _c(rows[:, 0], np.int32)
        head = _c(rows[:, 1], np.int32)
    n = tok.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    if num_threads is None:
        num_threads = os.cpu_count() or 1
    num_threads = max(1, min(int(num_threads), max(1, n)))
    rc = _load().orc_paged_attention_rows(
        _ptr(q, ctypes.c_uint16), t, hq, _ptr(kv_cache, ctypes.c_uint16), nb, bs, hkv, d,
        _ptr(bt, ctypes.c_int32), sl.shape[0], bt.shape[1] if bt.ndim == 2 else 0,
        _ptr(sl, ctypes.c_int32), _ptr(qsl, ctypes.c_int32), float(scale),
        _ptr(tok, ctypes.c_int32), _ptr(head, ctypes.c_int32), n, _ptr(out, ctypes.c_double), num_threads)
    _check(rc, "paged_attention")
    return out.reshape(t, hq, d) if rows is None else out
