"""Seeded synthetic inputs for paged-KV attention.

This module only draws random numbers and lays out the input structure that a
vLLM-style scheduler and KV-cache manager would hand to the attention layer
("Inside vLLM: Anatomy of a High-Throughput LLM Inference System", page 1,
"Scheduler" and "Prefix Caching"): per-request context lengths, new-token
counts, and block tables made of physical block ids drawn from a shuffled
pool. It holds none of the attention or KV-write arithmetic; both the CUDA
path and the CPU oracle read what it produces.

The workloads:

``tiny``       TinyLlama shape (32 q / 4 kv heads, head 64), 2 decode requests
               with contexts 17 and 40, a 64-block pool.
``tinyllama``  TinyLlama shape, 64 decode requests, contexts uniform in
               [128, 2048].
``llama8b``    Llama-3-8B shape (32 q / 8 kv heads, head 128), 256 decode
               requests, contexts uniform in [512, 4096].
``mixed``      Llama-3-8B shape, 4 chunked-prefill requests of 512 new tokens
               at prior offsets 0/512/1024/1536 plus 192 decode requests with
               contexts uniform in [256, 4096], shuffled into one ragged batch.
``prefix``     Llama-3-8B shape, 128 decode requests that share their first 64
               physical blocks (1024 tokens) and own a suffix of s tokens,
               s log-uniform in [64, 31744].
``specdec``    Llama-3-8B shape, 256 requests verifying 3 draft tokens each:
               4 new query tokens per request (speculative decoding scores
               k draft tokens plus one, "Speculative Decoding"; the pages'
               example sets num_speculative_tokens to 3), contexts uniform
               in [512, 4096].

Pools are 1.25x the blocks the batch needs (``tiny``: 64 blocks). Q, K, V and
the pool contents are N(0, 1) drawn in fp32 and rounded to bf16. Blocks that
no request references hold the bf16 bit pattern ``SENTINEL_BITS`` (a NaN).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
SENTINEL_BITS = 0xFFFF  # a bf16 NaN pattern
BASE_SEED = 20261202


@dataclass(frozen=True)
class ModelShape:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_size: int


TINYLLAMA = ModelShape("TinyLlama-1.1B", 32, 4, 64)
LLAMA3_8B = ModelShape("Llama-3-8B", 32, 8, 128)

WORKLOADS = ("tiny", "tinyllama", "llama8b", "mixed", "prefix", "specdec")


@dataclass
class Batch:
    """One flattened ragged batch and the pool it reads from."""

    workload: str
    shape: ModelShape
    seq_lens: np.ndarray          # int32 [R], context length including this step's tokens
    query_lens: np.ndarray        # int32 [R], new tokens of this step
    block_table: np.ndarray       # int32 [R][max_blocks_per_req], unused entries -1
    num_blocks: int
    seed: int
    shared_prefix_blocks: int = 0
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def query_start_loc(self) -> np.ndarray:
        qsl = np.zeros(self.num_reqs + 1, dtype=np.int32)
        np.cumsum(self.query_lens, out=qsl[1:])
        return qsl

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.shape.head_size)


def _ceil_div(a, b):
    return -(-a // b)


def _tables(rng, blocks_per_req, shared_blocks, pool_factor=1.25, num_blocks=None):
    """Block tables drawn from a shuffled pool: the first ``shared_blocks``
    entries of every table are the same physical blocks (a prefix-cache hit);
    every other entry is a block of its own."""
    blocks_per_req = np.asarray(blocks_per_req, dtype=np.int64)
    own = blocks_per_req - shared_blocks
    needed = int(shared_blocks + own.sum())
    if num_blocks is None:
        num_blocks = int(math.ceil(pool_factor * needed))
    assert needed <= num_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    mbr = int(blocks_per_req.max())
    table = np.full((blocks_per_req.shape[0], mbr), -1, dtype=np.int32)
    shared = perm[:shared_blocks]
    cursor = shared_blocks
    for r, nb in enumerate(blocks_per_req):
        table[r, :shared_blocks] = shared
        k = int(nb) - shared_blocks
        table[r, shared_blocks:nb] = perm[cursor:cursor + k]
        cursor += k
    return table, num_blocks


def make_batch(workload: str, seed_offset: int = 0) -> Batch:
    """The named workload. Its lengths and block tables are drawn with numpy's
    PCG64 generator from seed ``BASE_SEED + n + seed_offset``, where n is the
    workload's 1-based position in ``WORKLOADS`` (the configuration number:
    tiny 1, tinyllama 2, llama8b 3, mixed 4, prefix 5, specdec 6)."""
    idx = WORKLOADS.index(workload)
    seed = BASE_SEED + idx + 1 + seed_offset
    rng = np.random.Generator(np.random.PCG64(seed))
    bs = BLOCK_SIZE
    shared = 0
    if workload == "tiny":
        shape = TINYLLAMA
        seq = np.array([17, 40], dtype=np.int64)
        qlen = np.ones(2, dtype=np.int64)
        table, nb = _tables(rng, _ceil_div(seq, bs), 0, num_blocks=64)
        desc = "TinyLlama shape, 2 decode requests, contexts 17 and 40, 64-block pool"
    elif workload == "tinyllama":
        shape = TINYLLAMA
        seq = rng.integers(128, 2048, size=64, endpoint=True)
        qlen = np.ones(64, dtype=np.int64)
        table, nb = _tables(rng, _ceil_div(seq, bs), 0)
        desc = "TinyLlama shape, 64 decode requests, contexts U[128,2048]"
    elif workload == "llama8b":
        shape = LLAMA3_8B
        seq = rng.integers(512, 4096, size=256, endpoint=True)
        qlen = np.ones(256, dtype=np.int64)
        table, nb = _tables(rng, _ceil_div(seq, bs), 0)
        desc = "Llama-3-8B shape, 256 decode requests, contexts U[512,4096]"
    elif workload == "mixed":
        shape = LLAMA3_8B
        pre_seq = np.array([512, 1024, 1536, 2048], dtype=np.int64)
        pre_q = np.full(4, 512, dtype=np.int64)
        dec_seq = rng.integers(256, 4096, size=192, endpoint=True)
        dec_q = np.ones(192, dtype=np.int64)
        seq = np.concatenate([pre_seq, dec_seq])
        qlen = np.concatenate([pre_q, dec_q])
        order = rng.permutation(seq.shape[0])
        seq, qlen = seq[order], qlen[order]
        table, nb = _tables(rng, _ceil_div(seq, bs), 0)
        desc = ("Llama-3-8B shape, 4 chunked-prefill requests (512 new tokens at offsets "
                "0/512/1024/1536) + 192 decode requests with contexts U[256,4096], shuffled")
    elif workload == "prefix":
        shape = LLAMA3_8B
        shared = 64
        s = np.rint(np.exp(rng.uniform(math.log(64), math.log(31744), size=128))).astype(np.int64)
        seq = 1024 + s
        qlen = np.ones(128, dtype=np.int64)
        table, nb = _tables(rng, _ceil_div(seq, bs), shared)
        desc = ("Llama-3-8B shape, 128 decode requests sharing 64 prefix blocks (1024 tokens) "
                "+ log-uniform suffixes in [64, 31744]")
    elif workload == "specdec":
        shape = LLAMA3_8B
        seq = rng.integers(512, 4096, size=256, endpoint=True)
        qlen = np.full(256, 4, dtype=np.int64)
        table, nb = _tables(rng, _ceil_div(seq, bs), 0)
        desc = "Llama-3-8B shape, 256 requests verifying 3 draft tokens (4 query tokens each), contexts U[512,4096]"
    else:
        raise ValueError(f"unknown workload {workload!r}; expected one of {WORKLOADS}")
    return Batch(workload=workload, shape=shape, seq_lens=seq.astype(np.int32),
                 query_lens=qlen.astype(np.int32), block_table=table, num_blocks=int(nb),
                 seed=seed, shared_prefix_blocks=shared, description=desc)


def custom_batch(shape: ModelShape, seq_lens, query_lens, seed: int, shared_prefix_blocks: int = 0,
                 num_blocks: int | None = None, pool_factor: float = 1.25, workload: str = "custom") -> Batch:
    """A batch with caller-chosen lengths (edge cases in the tests)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seq = np.asarray(seq_lens, dtype=np.int64)
    qlen = np.asarray(query_lens, dtype=np.int64)
    nbr = np.maximum(_ceil_div(seq, BLOCK_SIZE), 1)
    table, nb = _tables(rng, nbr, shared_prefix_blocks, pool_factor=pool_factor, num_blocks=num_blocks)
    return Batch(workload=workload, shape=shape, seq_lens=seq.astype(np.int32),
                 query_lens=qlen.astype(np.int32), block_table=table, num_blocks=int(nb), seed=seed,
                 shared_prefix_blocks=shared_prefix_blocks, description="custom")


def _randn_bf16(shape, gen, device, chunk_elems=1 << 26):
    """N(0,1) in fp32, rounded to bf16, drawn in chunks to bound the fp32 scratch."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for start in range(0, n, chunk_elems):
        m = min(chunk_elems, n - start)
        flat[start:start + m] = torch.randn(m, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_tensors(batch: Batch, device="cpu", sentinel_unreferenced: bool = True) -> dict:
    """q [T][Hq][D], k/v [T][Hkv][D] (this step's new tokens) and the pool
    [NB][2][Hkv][16][D], all bf16, drawn from ``batch.seed`` on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(batch.seed)
    s = batch.shape
    t = batch.num_tokens
    q = _randn_bf16((t, s.num_q_heads, s.head_size), gen, device)
    k = _randn_bf16((t, s.num_kv_heads, s.head_size), gen, device)
    v = _randn_bf16((t, s.num_kv_heads, s.head_size), gen, device)
    pool = _randn_bf16((batch.num_blocks, 2, s.num_kv_heads, BLOCK_SIZE, s.head_size), gen, device)
    if sentinel_unreferenced:
        used = np.zeros(batch.num_blocks, dtype=bool)
        bt = batch.block_table
        used[bt[bt >= 0]] = True
        unused = torch.from_numpy(np.nonzero(~used)[0]).to(device)
        if unused.numel():
            pool.view(torch.int16)[unused] = np.int16(np.uint16(SENTINEL_BITS).view(np.int16))
    return {"q": q, "k": k, "v": v, "kv_cache": pool}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of a bf16 tensor's bits."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
