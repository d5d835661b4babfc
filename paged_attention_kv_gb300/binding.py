"""Thin Python binding over ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``).

Argument marshalling only: each function checks that the torch tensors it is
handed have the dtype, shape, device and contiguity the C call documents,
passes their device pointers and the current CUDA stream, and raises
``PagedKVError`` on a non-zero return code. Every step of the computation
runs in the library's CUDA kernels; there is no other code path. If the
library has not been built, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

BLOCK_SIZE = 16

# Return codes and device status bits (pagedkv.h).
PKV_OK = 0
PKV_E_NULL = -1
PKV_E_DIMS = -2
PKV_E_GQA = -3
PKV_E_BLOCK_SIZE = -4
PKV_E_HEAD_SIZE = -5
PKV_E_WORKSPACE = -6
PKV_E_ALIGN = -7
PKV_E_CUDA = -8
PKV_E_DEVICE = -9
PKV_DEV_BAD_QSL = 0x1
PKV_DEV_BAD_LEN = 0x2
PKV_DEV_BAD_BLOCK = 0x4
PKV_DEV_BAD_SLOT = 0x8
PKV_DEV_TIMEOUT = 0x10
PKV_DEV_OVERFLOW = 0x20

EXPORTED = ("pkv_kv_cache_bytes", "paged_slot_mapping", "paged_kv_write", "paged_kv_write_slots",
            "paged_kv_gather_blocks",
            "paged_kv_scatter_blocks", "paged_attention_workspace_bytes",
            "paged_attention_min_workspace_bytes", "paged_attention", "paged_attention_timed",
            "paged_attention_bounded", "paged_attention_static", "pkv_pipeline_create", "pkv_pipeline_next",
            "pkv_pipeline_submit", "pkv_pipeline_sync", "pkv_pipeline_destroy", "pkv_read_status", "pkv_selftest_bounded_wait", "pkv_status_string")


class PagedKVError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_size", ctypes.c_int32)]


PIPELINE_MAX_DEPTH = 4


class PipelineDesc(ctypes.Structure):
    """pkv_pipeline_desc of include/pagedkv.h."""
    _fields_ = [("depth", ctypes.c_int32), ("host_in", ctypes.c_void_p * PIPELINE_MAX_DEPTH),
                ("dev_in", ctypes.c_void_p * PIPELINE_MAX_DEPTH), ("in_bytes", ctypes.c_size_t),
                ("off_q", ctypes.c_size_t), ("off_k", ctypes.c_size_t), ("off_v", ctypes.c_size_t),
                ("off_block_table", ctypes.c_size_t), ("off_seq_lens", ctypes.c_size_t),
                ("off_query_start_loc", ctypes.c_size_t), ("num_tokens", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("max_num_reqs", ctypes.c_int32),
                ("max_blocks_per_req", ctypes.c_int32), ("cache", CacheDesc),
                ("slot_mapping", ctypes.c_void_p * PIPELINE_MAX_DEPTH), ("out", ctypes.c_void_p * PIPELINE_MAX_DEPTH),
                ("status", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("scale", ctypes.c_float), ("h2d_stream", ctypes.c_void_p), ("compute_stream", ctypes.c_void_p),
                ("d2h_stream", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    desc_p = ctypes.POINTER(CacheDesc)
    lib.pkv_kv_cache_bytes.argtypes = [desc_p, ctypes.POINTER(sz)]
    lib.paged_slot_mapping.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp]
    lib.paged_kv_write.argtypes = [vp, vp, vp, i32, vp, desc_p, vp, vp]
    lib.paged_kv_write_slots.argtypes = [vp, vp, vp, i32, i32, vp, vp, i32, vp, desc_p, vp, vp, vp]
    lib.paged_kv_gather_blocks.argtypes = [vp, desc_p, vp, i32, vp, vp, vp]
    lib.paged_kv_scatter_blocks.argtypes = [vp, vp, i32, vp, desc_p, vp, vp]
    lib.paged_attention_workspace_bytes.argtypes = [i32, i32, i32, desc_p, ctypes.POINTER(sz)]
    lib.paged_attention_min_workspace_bytes.argtypes = [i32, i32, i32, desc_p, ctypes.POINTER(sz)]
    lib.paged_attention.argtypes = [vp, i32, i32, vp, desc_p, vp, i32, i32, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.paged_attention_timed.argtypes = lib.paged_attention.argtypes + [ctypes.POINTER(vp)]
    lib.paged_attention_bounded.argtypes = [vp, i32, i32, vp, desc_p, vp, i32, i32, vp, vp, i32, ctypes.c_float, vp,
                                            vp, sz, vp, ctypes.POINTER(vp)]
    lib.paged_attention_static.argtypes = [vp, i32, i32, vp, desc_p, vp, i32, i32, vp, vp, ctypes.c_float, vp, vp]
    lib.pkv_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint32, vp]
    lib.pkv_pipeline_create.argtypes = [ctypes.POINTER(PipelineDesc), ctypes.POINTER(vp)]
    lib.pkv_pipeline_next.argtypes = [vp, ctypes.POINTER(i32)]
    lib.pkv_pipeline_submit.argtypes = [vp, i32, vp, vp, i32]
    lib.pkv_pipeline_sync.argtypes = [vp]
    lib.pkv_pipeline_destroy.argtypes = [vp]
    lib.pkv_read_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    return lib


LIB = _load()


def status_string(code: int) -> str:
    return LIB.pkv_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != PKV_OK:
        raise PagedKVError(rc, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _want(t: torch.Tensor, dtype, ndim, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def cache_desc(kv_cache: torch.Tensor) -> CacheDesc:
    """Descriptor of a pool tensor bf16 [num_blocks][2][num_kv_heads][16][head_size]."""
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2:
        raise ValueError(f"kv_cache must be [num_blocks][2][num_kv_heads][16][head_size], got {tuple(kv_cache.shape)}")
    nb, _, hkv, bs, d = kv_cache.shape
    return CacheDesc(nb, bs, hkv, d)


def pkv_kv_cache_bytes(num_blocks: int, num_kv_heads: int, head_size: int, block_size: int = BLOCK_SIZE) -> int:
    out = ctypes.c_size_t(0)
    _check(LIB.pkv_kv_cache_bytes(ctypes.byref(CacheDesc(num_blocks, block_size, num_kv_heads, head_size)),
                                  ctypes.byref(out)), "pkv_kv_cache_bytes")
    return out.value


def paged_slot_mapping(block_table, seq_lens, query_start_loc, num_tokens: int, num_blocks: int,
                       slot_mapping=None, status=None, stream=None) -> torch.Tensor:
    _want(block_table, torch.int32, 2, "block_table")
    _want(seq_lens, torch.int32, 1, "seq_lens")
    _want(query_start_loc, torch.int32, 1, "query_start_loc")
    num_reqs = seq_lens.shape[0]
    if query_start_loc.shape[0] != num_reqs + 1 or block_table.shape[0] != num_reqs:
        raise ValueError("block_table, seq_lens and query_start_loc disagree on the number of requests")
    if slot_mapping is None:
        slot_mapping = torch.empty(num_tokens, dtype=torch.int32, device=seq_lens.device)
    _want(slot_mapping, torch.int32, 1, "slot_mapping")
    if slot_mapping.shape[0] < num_tokens:
        raise ValueError("slot_mapping is shorter than num_tokens")
    _check(LIB.paged_slot_mapping(_ptr(block_table), num_reqs, block_table.shape[1], _ptr(seq_lens),
                                  _ptr(query_start_loc), num_tokens, num_blocks, _ptr(slot_mapping), _ptr(status),
                                  _stream(stream)), "paged_slot_mapping")
    return slot_mapping


def paged_kv_write(k, v, slot_mapping, kv_cache, status=None, stream=None) -> None:
    _want(k, torch.bfloat16, 3, "k")
    _want(v, torch.bfloat16, 3, "v")
    _want(slot_mapping, torch.int32, 1, "slot_mapping")
    _want(kv_cache, torch.bfloat16, 5, "kv_cache")
    desc = cache_desc(kv_cache)
    t = k.shape[0]
    if v.shape != k.shape or k.shape[1] != desc.num_kv_heads or k.shape[2] != desc.head_size:
        raise ValueError("k/v must be [num_tokens][num_kv_heads][head_size] matching kv_cache")
    if slot_mapping.shape[0] < t:
        raise ValueError("slot_mapping is shorter than k")
    _check(LIB.paged_kv_write(_ptr(k), _ptr(v), _ptr(slot_mapping), t, _ptr(kv_cache), ctypes.byref(desc),
                              _ptr(status), _stream(stream)), "paged_kv_write")


def block_bytes(kv_cache: torch.Tensor) -> int:
    d = cache_desc(kv_cache)
    return 2 * d.block_size * d.num_kv_heads * d.head_size * 2


def paged_kv_gather_blocks(kv_cache, block_ids, staging=None, status=None, stream=None) -> torch.Tensor:
    """staging[i] = pool block block_ids[i]; staging is uint8 [n][block_bytes]."""
    _want(kv_cache, torch.bfloat16, 5, "kv_cache")
    _want(block_ids, torch.int32, 1, "block_ids")
    n = block_ids.shape[0]
    if staging is None:
        staging = torch.empty((n, block_bytes(kv_cache)), dtype=torch.uint8, device=kv_cache.device)
    _want(staging, torch.uint8, 2, "staging")
    if staging.shape[0] < n or staging.shape[1] != block_bytes(kv_cache):
        raise ValueError("staging must be [num_ids][block_bytes] bytes")
    desc = cache_desc(kv_cache)
    _check(LIB.paged_kv_gather_blocks(_ptr(kv_cache), ctypes.byref(desc), _ptr(block_ids), n, _ptr(staging),
                                      _ptr(status), _stream(stream)), "paged_kv_gather_blocks")
    return staging


def paged_kv_scatter_blocks(staging, block_ids, kv_cache, status=None, stream=None) -> None:
    """pool block block_ids[i] = staging[i]."""
    _want(kv_cache, torch.bfloat16, 5, "kv_cache")
    _want(block_ids, torch.int32, 1, "block_ids")
    _want(staging, torch.uint8, 2, "staging")
    n = block_ids.shape[0]
    if staging.shape[0] < n or staging.shape[1] != block_bytes(kv_cache):
        raise ValueError("staging must be [num_ids][block_bytes] bytes")
    desc = cache_desc(kv_cache)
    _check(LIB.paged_kv_scatter_blocks(_ptr(staging), _ptr(block_ids), n, _ptr(kv_cache), ctypes.byref(desc),
                                       _ptr(status), _stream(stream)), "paged_kv_scatter_blocks")


def paged_attention_workspace_bytes(max_num_reqs: int, max_num_tokens: int, num_q_heads: int, num_blocks: int,
                                    num_kv_heads: int, head_size: int) -> int:
    out = ctypes.c_size_t(0)
    desc = CacheDesc(num_blocks, BLOCK_SIZE, num_kv_heads, head_size)
    _check(LIB.paged_attention_workspace_bytes(max_num_reqs, max_num_tokens, num_q_heads, ctypes.byref(desc),
                                               ctypes.byref(out)), "paged_attention_workspace_bytes")
    return out.value


def paged_attention_min_workspace_bytes(max_num_reqs: int, max_num_tokens: int, num_q_heads: int,
                                        num_blocks: int, num_kv_heads: int, head_size: int) -> int:
    out = ctypes.c_size_t(0)
    desc = CacheDesc(num_blocks, BLOCK_SIZE, num_kv_heads, head_size)
    _check(LIB.paged_attention_min_workspace_bytes(max_num_reqs, max_num_tokens, num_q_heads, ctypes.byref(desc),
                                                   ctypes.byref(out)), "paged_attention_min_workspace_bytes")
    return out.value


def alloc_workspace(max_num_reqs: int, max_num_tokens: int, num_q_heads: int, kv_cache: torch.Tensor) -> torch.Tensor:
    d = cache_desc(kv_cache)
    nbytes = paged_attention_workspace_bytes(max_num_reqs, max_num_tokens, num_q_heads, d.num_blocks,
                                             d.num_kv_heads, d.head_size)
    # int64 elements: torch's caching allocator returns 512-byte aligned blocks
    return torch.empty((nbytes + 7) // 8, dtype=torch.int64, device=kv_cache.device)


def paged_attention(q, kv_cache, block_table, seq_lens, query_start_loc, scale: float, out=None, workspace=None,
                    stream=None, events=None, max_query_len: int = 0) -> torch.Tensor:
    """Attention over the paged pool. ``events``: optional four
    torch.cuda.Event(enable_timing=True) recorded before the work-list
    kernel, after it, after the chunk-tile kernel and after the split-KV
    kernel. ``max_query_len``: optional bound on any request's new tokens
    (0: none); below 128 / GQA group the chunk-tile kernel is not launched."""
    _want(q, torch.bfloat16, 3, "q")
    _want(kv_cache, torch.bfloat16, 5, "kv_cache")
    _want(block_table, torch.int32, 2, "block_table")
    _want(seq_lens, torch.int32, 1, "seq_lens")
    _want(query_start_loc, torch.int32, 1, "query_start_loc")
    desc = cache_desc(kv_cache)
    t, hq, d = q.shape
    num_reqs = seq_lens.shape[0]
    if d != desc.head_size:
        raise ValueError("q head_size differs from kv_cache")
    if query_start_loc.shape[0] != num_reqs + 1 or block_table.shape[0] != num_reqs:
        raise ValueError("block_table, seq_lens and query_start_loc disagree on the number of requests")
    if out is None:
        out = torch.empty_like(q)
    _want(out, torch.bfloat16, 3, "out")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = alloc_workspace(num_reqs, t, hq, kv_cache)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    args = (_ptr(q), t, hq, _ptr(kv_cache), ctypes.byref(desc), _ptr(block_table), num_reqs, block_table.shape[1],
            _ptr(seq_lens), _ptr(query_start_loc), float(scale), _ptr(out), _ptr(workspace), nbytes, _stream(stream))
    if max_query_len:
        head, tail = args[:10], args[10:]
        handles = None
        if events is not None:
            handles = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(_event_handle(e, stream)) for e in events])
        _check(LIB.paged_attention_bounded(*head, int(max_query_len), *tail, handles), "paged_attention_bounded")
    elif events is None:
        _check(LIB.paged_attention(*args), "paged_attention")
    else:
        handles = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(_event_handle(e, stream)) for e in events])
        _check(LIB.paged_attention_timed(*args, handles), "paged_attention_timed")
    return out


def paged_attention_static(q, kv_cache, block_table, seq_lens, query_start_loc, scale: float, out,
                           stream=None) -> torch.Tensor:
    """paged_attention without a workspace: for callers that cannot allocate
    device memory when they run attention (the library's fixed 16 MiB scratch
    array is used instead). ``out`` must be preallocated. Calls on one
    device share that array, so they must not overlap on the GPU."""
    _want(q, torch.bfloat16, 3, "q")
    _want(kv_cache, torch.bfloat16, 5, "kv_cache")
    _want(block_table, torch.int32, 2, "block_table")
    _want(seq_lens, torch.int32, 1, "seq_lens")
    _want(query_start_loc, torch.int32, 1, "query_start_loc")
    _want(out, torch.bfloat16, 3, "out")
    desc = cache_desc(kv_cache)
    t, hq, _ = q.shape
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    _check(LIB.paged_attention_static(_ptr(q), t, hq, _ptr(kv_cache), ctypes.byref(desc), _ptr(block_table),
                                      seq_lens.shape[0], block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
                                      float(scale), _ptr(out), _stream(stream)), "paged_attention_static")
    return out


def _event_handle(ev, stream) -> int:
    """Raw cudaEvent_t of a torch.cuda.Event (torch creates it on first record)."""
    if ev is None:
        return 0
    if not ev.cuda_event:
        ev.record(stream if stream is not None else torch.cuda.current_stream())
    return int(ev.cuda_event)


def pkv_selftest_bounded_wait(status: torch.Tensor, timeout_us: int = 2000, stream=None) -> None:
    """Run the bounded-wait self-test: a wait on an mbarrier nothing arrives
    on gives up after ``timeout_us`` and ORs PKV_DEV_TIMEOUT into ``status``."""
    _want(status, torch.int32, 1, "status")
    _check(LIB.pkv_selftest_bounded_wait(_ptr(status), int(timeout_us), _stream(stream)), "pkv_selftest_bounded_wait")


def pkv_read_status(status: torch.Tensor, stream=None) -> int:
    """Device status word (synchronises the stream). For paged_attention pass
    its workspace: the word is the workspace's first 4 bytes."""
    v = ctypes.c_int32(0)
    rc = LIB.pkv_read_status(_ptr(status), _stream(stream), ctypes.byref(v))
    if rc not in (PKV_OK, PKV_E_DEVICE):
        _check(rc, "pkv_read_status")
    return v.value


class StepBuffers:
    """Device buffers of one paged-attention step for a fixed batch: the
    metadata tables, slot mapping, output, workspace and status word."""

    def __init__(self, batch, tensors: dict):
        dev = tensors["q"].device
        self.batch = batch
        self.q = tensors["q"]
        self.k = tensors["k"]
        self.v = tensors["v"]
        self.kv_cache = tensors["kv_cache"]
        self.block_table = torch.from_numpy(batch.block_table).to(dev)
        self.seq_lens = torch.from_numpy(batch.seq_lens).to(dev)
        self.query_start_loc = torch.from_numpy(batch.query_start_loc).to(dev)
        self.num_tokens = batch.num_tokens
        # the longest request's new tokens, known to the scheduler that built the batch
        self.max_query_len = int(batch.query_lens.max()) if batch.num_reqs else 0
        self.slot_mapping = torch.empty(self.num_tokens, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.workspace = alloc_workspace(batch.num_reqs, self.num_tokens, batch.shape.num_q_heads, self.kv_cache)

    def prepared(self, stream=None) -> "PreparedStep":
        """This step's calls with their C arguments built once (for
        loops that enqueue the same step many times: the per-call checks and
        argument conversion of the wrappers cost the host more than a small
        step costs the GPU). Valid while these buffers stay in place."""
        return PreparedStep(self, stream)

    def step(self, stream=None):
        """Slot mapping, KV write and attention, enqueued on `stream`."""
        paged_slot_mapping(self.block_table, self.seq_lens, self.query_start_loc, self.num_tokens,
                           self.batch.num_blocks, self.slot_mapping, self.status, stream)
        paged_kv_write(self.k, self.v, self.slot_mapping, self.kv_cache, self.status, stream)
        paged_attention(self.q, self.kv_cache, self.block_table, self.seq_lens, self.query_start_loc,
                        self.batch.scale, self.out, self.workspace, stream, max_query_len=self.max_query_len)
        return self.out


class PreparedStep:
    """Slot mapping, KV write and attention of a StepBuffers, checked once,
    then enqueued by calling the object: two C calls (the fused slot mapping
    and KV write, then attention) with prebuilt arguments and no per-call
    Python checks."""

    def __init__(self, buf: "StepBuffers", stream=None):
        for t, dt, nd, name in ((buf.q, torch.bfloat16, 3, "q"), (buf.k, torch.bfloat16, 3, "k"),
                                (buf.v, torch.bfloat16, 3, "v"), (buf.kv_cache, torch.bfloat16, 5, "kv_cache"),
                                (buf.block_table, torch.int32, 2, "block_table"),
                                (buf.seq_lens, torch.int32, 1, "seq_lens"),
                                (buf.query_start_loc, torch.int32, 1, "query_start_loc"),
                                (buf.slot_mapping, torch.int32, 1, "slot_mapping"),
                                (buf.status, torch.int32, 1, "status"), (buf.out, torch.bfloat16, 3, "out")):
            _want(t, dt, nd, name)
        if not buf.workspace.is_cuda or not buf.workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        b = buf.batch
        self.desc = cache_desc(buf.kv_cache)  # kept alive: passed by reference
        t, hq, _ = buf.q.shape
        r = b.num_reqs
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        st = _stream(stream)
        desc = ctypes.byref(self.desc)
        ws_bytes = ctypes.c_size_t(buf.workspace.numel() * buf.workspace.element_size())
        if buf.k.shape[0] != buf.num_tokens:
            raise ValueError("k must hold the step's num_tokens rows")
        self.calls = (
            ("paged_kv_write_slots", LIB.paged_kv_write_slots,
             (_ptr(buf.k), _ptr(buf.v), _ptr(buf.block_table), i32(r), i32(buf.block_table.shape[1]),
              _ptr(buf.seq_lens), _ptr(buf.query_start_loc), i32(buf.num_tokens), _ptr(buf.kv_cache), desc,
              _ptr(buf.slot_mapping), _ptr(buf.status), st)),
            ("paged_attention_bounded", LIB.paged_attention_bounded,
             (_ptr(buf.q), i32(t), i32(hq), _ptr(buf.kv_cache), desc, _ptr(buf.block_table), i32(r),
              i32(buf.block_table.shape[1]), _ptr(buf.seq_lens), _ptr(buf.query_start_loc),
              i32(buf.max_query_len), ctypes.c_float(b.scale), _ptr(buf.out), _ptr(buf.workspace), ws_bytes, st,
              None)),
        )
        self.buf = buf  # keeps the tensors alive

    def __call__(self) -> None:
        for name, fn, args in self.calls:
            rc = fn(*args)
            if rc != PKV_OK:
                raise PagedKVError(rc, name)


class StepGraph:
    """One step (slot mapping, KV write, attention) captured into a CUDA
    graph and replayed: the launches of a step cost one graph launch. The
    graph keeps the buffers' device addresses, so new inputs of the same
    shape are copied into ``buffers`` before each replay (the engine loop
    of the pages captures one graph per warm-up batch size in the same way,
    page 1, "LLM Engine constructor", KV-cache initialisation)."""

    def __init__(self, buffers: StepBuffers):
        self.buffers = buffers
        # first calls set up the device (kernel attributes, entry points)
        # and must run outside capture
        buffers.step()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            buffers.step()
        torch.cuda.synchronize()

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.buffers.out


class HostStepPipeline:
    """Steps whose inputs (q, k, v and the metadata tables) come from host
    memory and whose output goes back to host memory.

    Each step's inputs sit in one packed pinned host buffer and cross to the
    device in ONE copy; the output returns in one copy. ``depth`` slots
    alternate: step i+1's host-to-device copy runs on one copy stream while
    step i computes, and step i's output returns on a second copy stream
    while step i+1 computes. Each step is the same three calls as
    ``StepBuffers.step`` (slot mapping, KV write, attention) on the compute
    stream, so steps still run in order against the pool. The copies, the
    calls and the events that order them are the library's native pipeline
    (``pkv_pipeline_*``, one C call per step); the buffers and streams are
    PyTorch's.

    Use: ``inp = pipe.next_inputs()`` (host views q, k, v, block_table,
    seq_lens, query_start_loc of the next slot; waits until that slot's
    previous copy has left), fill them, then ``pipe.submit(out_host)``. The
    step's ``out_host`` is complete after ``synchronize()`` or after the
    event ``submit`` returns.
    """

    def __init__(self, kv_cache: torch.Tensor, max_num_reqs: int, num_tokens: int, max_blocks_per_req: int,
                 num_q_heads: int, scale: float, depth: int = 2, compute_stream=None):
        dev = kv_cache.device
        d = cache_desc(kv_cache)
        self.kv_cache = kv_cache
        self.scale = float(scale)
        self.num_tokens = int(num_tokens)
        self.num_blocks = int(d.num_blocks)
        self.max_num_reqs = int(max_num_reqs)
        self.depth = int(depth)
        self.compute = compute_stream or torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        T, Hq, Hkv, D = self.num_tokens, int(num_q_heads), int(d.num_kv_heads), int(d.head_size)
        R, M = self.max_num_reqs, int(max_blocks_per_req)
        # packed layout: (name, dtype, shape), each array 256-byte aligned
        spec = [("q", torch.bfloat16, (T, Hq, D)), ("k", torch.bfloat16, (T, Hkv, D)),
                ("v", torch.bfloat16, (T, Hkv, D)), ("block_table", torch.int32, (R, M)),
                ("seq_lens", torch.int32, (R,)), ("query_start_loc", torch.int32, (R + 1,))]
        offs, off = [], 0
        for _, dt, shp in spec:
            n = 1
            for x in shp:
                n *= x
            offs.append(off)
            off += -(-n * torch.tensor([], dtype=dt).element_size() // 256) * 256
        self.packed_bytes = off

        def views(raw):
            out = {}
            for (name, dt, shp), o in zip(spec, offs):
                n = 1
                for x in shp:
                    n *= x
                size = torch.tensor([], dtype=dt).element_size()
                out[name] = raw[o:o + n * size].view(dt).view(shp)
            return out

        self.host_raw = [torch.empty(off, dtype=torch.uint8, pin_memory=True) for _ in range(self.depth)]
        self.dev_raw = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(self.depth)]
        self.host_in = [views(r) for r in self.host_raw]
        self.dev_in = [views(r) for r in self.dev_raw]
        self.slot_mapping = [torch.empty(T, dtype=torch.int32, device=dev) for _ in range(self.depth)]
        self.out = [torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev) for _ in range(self.depth)]
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = alloc_workspace(R, self.num_tokens, Hq, kv_cache)
        if not 1 <= self.depth <= PIPELINE_MAX_DEPTH:
            raise PagedKVError(PKV_E_DIMS, "pipeline depth outside 1..4")
        desc = PipelineDesc()
        desc.depth = self.depth
        for i in range(self.depth):
            desc.host_in[i] = self.host_raw[i].data_ptr()
            desc.dev_in[i] = self.dev_raw[i].data_ptr()
            desc.slot_mapping[i] = self.slot_mapping[i].data_ptr()
            desc.out[i] = self.out[i].data_ptr()
        desc.in_bytes = off
        desc.off_q, desc.off_k, desc.off_v, desc.off_block_table, desc.off_seq_lens, desc.off_query_start_loc = offs
        desc.num_tokens, desc.num_q_heads, desc.max_num_reqs, desc.max_blocks_per_req = T, Hq, R, M
        desc.cache = d
        desc.status = self.status.data_ptr()
        desc.workspace = self.workspace.data_ptr()
        desc.workspace_bytes = self.workspace.numel() * self.workspace.element_size()
        desc.scale = self.scale
        desc.h2d_stream = self.h2d.cuda_stream
        desc.compute_stream = self.compute.cuda_stream
        desc.d2h_stream = self.d2h.cuda_stream
        self._desc = desc
        handle = ctypes.c_void_p(0)
        _check(LIB.pkv_pipeline_create(ctypes.byref(desc), ctypes.byref(handle)), "pkv_pipeline_create")
        self._handle = handle
        self._lib = LIB
        self._slot = ctypes.c_int32(0)
        self.i = 0

    def __del__(self):
        handle = getattr(self, "_handle", None)
        if handle is not None and handle.value:
            self._lib.pkv_pipeline_destroy(handle)
            self._handle = None

    def slot_inputs(self, slot: int) -> dict:
        """Host views of one slot, for filling every slot before the first
        step (no waiting: call it only while no step is in flight)."""
        return self.host_in[slot]

    def next_inputs(self) -> dict:
        """Host views to fill with the next step's inputs (waits until that
        slot's previous input copy has been read)."""
        _check(LIB.pkv_pipeline_next(self._handle, ctypes.byref(self._slot)), "pkv_pipeline_next")
        return self.host_in[self._slot.value]

    def submit(self, out_host: torch.Tensor, num_reqs: int | None = None, kv_cache=None,
               max_query_len: int | None = None) -> None:
        """Enqueue the step whose inputs are in ``next_inputs()`` (one C call:
        the input copy, the three calls and the output copy, ordered by the
        pipeline's events). ``num_reqs``: the requests of this step (default:
        all). ``kv_cache``: this step's pool when it is not the one the
        pipeline was built with (another layer's pool of the same shape).
        ``max_query_len``: the longest request of the step, as the scheduler
        knows it (default: taken from the host copy of query_start_loc).
        ``out_host`` (pinned, the output's shape) holds the output after
        ``synchronize()``."""
        pool = self.kv_cache if kv_cache is None else kv_cache
        if pool.shape != self.kv_cache.shape or pool.dtype != self.kv_cache.dtype:
            raise PagedKVError(PKV_E_DIMS, "kv_cache differs in shape from the pipeline's pool")
        if out_host.numel() * out_host.element_size() != self.out[0].numel() * self.out[0].element_size():
            raise PagedKVError(PKV_E_DIMS, "out_host differs in size from the step's output")
        R = self.max_num_reqs if num_reqs is None else int(num_reqs)
        mq = -1 if max_query_len is None else max(0, int(max_query_len))
        _check(LIB.pkv_pipeline_submit(self._handle, R, pool.data_ptr(), out_host.data_ptr(), mq),
               "pkv_pipeline_submit")
        self.i += 1

    def synchronize(self) -> None:
        _check(LIB.pkv_pipeline_sync(self._handle), "pkv_pipeline_sync")

    def read_status(self) -> tuple[int, int]:
        """(slot mapping / KV write status, attention status)."""
        self.synchronize()
        return pkv_read_status(self.status, self.compute), pkv_read_status(self.workspace, self.compute)


def run_step(batch, tensors: dict, stream=None) -> dict:
    """One step on device tensors; raises if a device status bit is set."""
    buf = StepBuffers(batch, tensors)
    buf.step(stream)
    st = pkv_read_status(buf.status, stream)
    wst = pkv_read_status(buf.workspace, stream)
    if st or wst:
        raise PagedKVError(PKV_E_DEVICE, f"device status {st:#x} (slot/write) {wst:#x} (attention)")
    return {"slot_mapping": buf.slot_mapping, "kv_cache": buf.kv_cache, "out": buf.out, "buffers": buf}
