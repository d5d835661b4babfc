"""GPU parity at the size limits of the work-list kernel and the split-KV path.

The work-list kernel keeps its per-request tables in shared memory up to 4096
requests and its per-group tables up to 8192 decode groups; past either it
keeps them in the workspace and waits for the previous kernel before it
starts. These batches cross each limit, alone and with a shared prefix, and
one request runs at a 128k-token context. Outputs are compared with the fp64
oracle on sampled rows (every row of the long request), slot mapping and the
pool bit for bit.
"""
import numpy as np
import pytest
import torch

from paged_attention_kv_gb300 import workloads as wl

from parity_utils import assert_attention_close, device_tensors, host_inputs, oracle_step, run_gpu_step

pytestmark = pytest.mark.gpu

LLAMA = wl.LLAMA3_8B
TINY = wl.TINYLLAMA


def _rows(batch, n, seed, extra_tokens=()):
    rng = np.random.default_rng(seed)
    t = rng.integers(0, batch.num_tokens, size=n)
    h = rng.integers(0, batch.shape.num_q_heads, size=n)
    rows = [np.stack([t, h], axis=1)]
    for tok in extra_tokens:
        hs = np.arange(batch.shape.num_q_heads)
        rows.append(np.stack([np.full_like(hs, tok), hs], axis=1))
    return np.concatenate(rows).astype(np.int64)


def _check_sampled(batch, rows, ten=None):
    ten = ten if ten is not None else device_tensors(batch)
    host = host_inputs(ten)
    slots, pool, ref = oracle_step(batch, host, rows=rows)
    buf, st, wst = run_gpu_step(batch, ten)
    assert st == 0 and wst == 0, (hex(st), hex(wst))
    assert np.array_equal(buf.slot_mapping.cpu().numpy(), slots)
    assert np.array_equal(wl.bf16_bits(buf.kv_cache), pool)
    assert_attention_close(buf.out, ref, rows=rows, what=batch.workload)
    return buf


def _record(buf):
    h = buf.workspace[:8].view(torch.int32).cpu().numpy()
    return {"n_groups": int(h[3]), "cascade_blocks": int(h[10])}


def test_more_requests_than_the_shared_memory_tables():
    """5000 decode requests (> 4096): per-request tables in the workspace."""
    rng = np.random.default_rng(501)
    seq = rng.integers(1, 200, size=5000)
    batch = wl.custom_batch(TINY, seq, np.ones(5000, np.int64), 502)
    buf = _check_sampled(batch, _rows(batch, 3000, 503, extra_tokens=(0, 4999)))
    assert _record(buf)["n_groups"] == 5000


def test_more_requests_than_the_tables_with_a_shared_prefix():
    """4500 decode requests sharing 4 blocks: the prefix tiles run from the
    workspace-table path too (the full workspace holds two partial slots per
    query row)."""
    rng = np.random.default_rng(511)
    seq = 64 + rng.integers(1, 150, size=4500)
    batch = wl.custom_batch(LLAMA, seq, np.ones(4500, np.int64), 512, shared_prefix_blocks=4)
    buf = _check_sampled(batch, _rows(batch, 3000, 513, extra_tokens=(0, 4499)))
    assert _record(buf)["cascade_blocks"] == 4


def test_more_query_rows_than_the_shared_memory_group_tables():
    """20 chunked-prefill requests of 820 tokens plus 50 decode requests at
    GQA 8: 8225 + 70 decode-group slots (> 8192), chunk tiles for the
    prefill rows."""
    rng = np.random.default_rng(521)
    pre_n = np.full(20, 820)
    pre_seq = pre_n + rng.integers(0, 600, size=20)
    dec_seq = rng.integers(16, 3000, size=50)
    seq = np.concatenate([pre_seq, dec_seq])
    ql = np.concatenate([pre_n, np.ones(50, np.int64)])
    order = rng.permutation(seq.shape[0])
    batch = wl.custom_batch(TINY, seq[order], ql[order], 522)
    qsl = batch.query_start_loc
    last_tokens = [int(qsl[r + 1]) - 1 for r in range(batch.num_reqs)]
    _check_sampled(batch, _rows(batch, 3000, 523, extra_tokens=last_tokens[:8]))


def test_a_128k_token_context():
    """One decode request at 131072 tokens (8192 blocks, many splits) among
    short ones; every row of the long request is checked."""
    seq = np.array([37, 131072, 500, 16], np.int64)
    batch = wl.custom_batch(LLAMA, seq, np.ones(4, np.int64), 531, pool_factor=1.05)
    _check_sampled(batch, _rows(batch, 64, 532, extra_tokens=(0, 1, 2, 3)))
