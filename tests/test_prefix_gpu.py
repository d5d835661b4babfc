"""GPU parity of the shared-prefix path ("Inside vLLM", page 1, "Prefix
Caching": requests whose block-aligned prefix is cached reuse the same
physical blocks).

When every request's block table starts with the same P >= 4 blocks and
those keys are visible to every query row, the split-KV kernel also runs
"prefix tiles": 16 query rows at a time, across request boundaries, against
the shared blocks only, merged with each tile's own splits. These tests
check that the pass runs when it should (the plan's record in the workspace
header), stays off when it must, and that the outputs match the oracle
either way.
"""
import numpy as np
import pytest
import torch

from paged_attention_kv_gb300 import binding as pkv
from paged_attention_kv_gb300 import workloads as wl

from parity_utils import assert_attention_close, device_tensors, host_inputs, oracle_step, run_gpu_step

pytestmark = pytest.mark.gpu

LLAMA = wl.LLAMA3_8B
TINY = wl.TINYLLAMA


def plan_record(buf):
    """The plan kernel's record at the head of the workspace (int32 words:
    status, n_items, split_blocks, n_groups, n_partial_rows, next_item,
    n_chunk_items, next_chunk_item, diag, n_prefix_items, cascade_blocks)."""
    h = buf.workspace[:8].view(torch.int32).cpu().numpy()
    return {"n_items": int(h[1]), "split_blocks": int(h[2]), "n_prefix_items": int(h[9]),
            "cascade_blocks": int(h[10])}


def _run(batch, ten=None, workspace_bytes=None):
    ten = ten if ten is not None else device_tensors(batch, generate_on="cpu")
    host = host_inputs(ten)
    slots, pool, ref = oracle_step(batch, host)
    buf, st, wst = run_gpu_step(batch, ten, workspace_bytes)
    assert st == 0 and wst == 0, (hex(st), hex(wst))
    assert np.array_equal(buf.slot_mapping.cpu().numpy(), slots)
    assert np.array_equal(wl.bf16_bits(buf.kv_cache), pool)
    assert_attention_close(buf.out, ref, what=batch.workload)
    return buf, ref


def _prefix_tiles(batch):
    g = batch.shape.num_q_heads // batch.shape.num_kv_heads
    return -(-batch.num_tokens * g // 16) * batch.shape.num_kv_heads


def test_prefix_workload_runs_the_shared_pass():
    """128 decode requests sharing 64 blocks: P = 64, one prefix tile per 16
    rows and kv head, outputs within tolerance of the oracle."""
    batch = wl.make_batch("prefix")
    buf, _ = _run(batch, device_tensors(batch))
    rec = plan_record(buf)
    assert rec["cascade_blocks"] == 64
    assert rec["n_prefix_items"] == _prefix_tiles(batch)


@pytest.mark.parametrize("shape,ql", [
    (LLAMA, [1] * 6),
    (LLAMA, [4, 4, 4, 4, 4]),              # speculative verify: 16-row tiles, one request each
    (LLAMA, [1, 3, 5, 2, 7, 1, 2]),        # decode tiles straddling prefix tiles
    (TINY, [2, 1, 9, 1, 1]),               # head 64, GQA 8
    (wl.ModelShape("h12-4-128", 12, 4, 128), [1, 2, 3, 4, 5]),   # GQA 3: 16 rows hold partial tokens
    (wl.ModelShape("h8-8-64", 8, 8, 64), [1, 1, 1, 1, 1, 1, 1, 1, 1]),  # no GQA: one row per token
], ids=["decode", "specdec", "ragged", "d64", "gqa3", "mha"])
def test_shared_prefix_with_ragged_queries(shape, ql):
    shared = 8
    rng = np.random.default_rng(len(ql) * 31 + shape.head_size)
    suffix = rng.integers(1, 600, size=len(ql))
    seq = shared * 16 + suffix + np.asarray(ql)
    batch = wl.custom_batch(shape, seq, ql, 400 + len(ql) + shape.num_q_heads, shared_prefix_blocks=shared)
    buf, _ = _run(batch)
    rec = plan_record(buf)
    assert rec["cascade_blocks"] == shared
    assert rec["n_prefix_items"] == _prefix_tiles(batch)


def test_prefix_is_capped_by_the_shortest_visible_context():
    """A request whose new tokens start inside the shared blocks: only the
    blocks every row sees whole go to the shared pass (P = 6 of 8)."""
    shared = 8
    seq = [shared * 16 + 300, shared * 16 + 2, shared * 16 + 40, shared * 16 + 900]
    ql = [1, 20, 1, 1]     # request 1: its first row sees keys [0, 111), 6.9 blocks
    batch = wl.custom_batch(LLAMA, seq, ql, 410, shared_prefix_blocks=shared)
    buf, _ = _run(batch)
    assert plan_record(buf)["cascade_blocks"] == (seq[1] - ql[1]) // 16


@pytest.mark.parametrize("case", ["three_requests", "short_prefix", "chunk_request", "no_sharing"])
def test_shared_pass_stays_off(case):
    """The pass needs >= 4 requests, >= 4 shared blocks, and split-KV rows
    only; otherwise the batch runs as before."""
    seq, ql, shared = [400, 900, 333, 1500, 171], [1, 1, 2, 1, 1], 8
    if case == "three_requests":
        seq, ql = seq[:3], ql[:3]
    elif case == "short_prefix":
        shared = 3
    elif case == "chunk_request":
        seq[3], ql[3] = 1500, 64          # 256 rows: a tensor-core chunk request
    elif case == "no_sharing":
        shared = 0
    batch = wl.custom_batch(LLAMA, seq, ql, 420, shared_prefix_blocks=shared)
    buf, _ = _run(batch)
    rec = plan_record(buf)
    assert rec["cascade_blocks"] == 0 and rec["n_prefix_items"] == 0


def test_shared_pass_dropped_when_partials_do_not_fit():
    """With the minimal workspace there is no room for partial rows: the
    plan drops the shared pass and every tile runs unsplit."""
    batch = wl.custom_batch(LLAMA, [200, 700, 1300, 450, 129], [1, 1, 1, 2, 1], 430, shared_prefix_blocks=8)
    s = batch.shape
    minimal = pkv.paged_attention_min_workspace_bytes(batch.num_reqs, batch.num_tokens, s.num_q_heads,
                                                      batch.num_blocks, s.num_kv_heads, s.head_size)
    buf, _ = _run(batch, workspace_bytes=minimal)
    assert plan_record(buf)["cascade_blocks"] == 0


def test_identical_requests_give_identical_bits():
    """Two requests with the same block table, the same context and the same
    query give the same output bits, wherever their rows fall in the prefix
    tiles."""
    shared = 16
    seq, ql = [shared * 16 + 500, shared * 16 + 77, shared * 16 + 500, shared * 16 + 1000, shared * 16 + 9], [1] * 5
    batch = wl.custom_batch(LLAMA, seq, ql, 440, shared_prefix_blocks=shared)
    batch.block_table[2] = batch.block_table[0]
    ten = device_tensors(batch, generate_on="cpu")
    ten["q"][2] = ten["q"][0]
    ten["k"][2] = ten["k"][0]
    ten["v"][2] = ten["v"][0]
    buf, _ = _run(batch, ten)
    assert plan_record(buf)["cascade_blocks"] == shared
    assert torch.equal(buf.out[0].view(torch.int16), buf.out[2].view(torch.int16))


def test_requests_without_new_tokens_in_a_shared_batch():
    shared = 6
    seq = [shared * 16 + x for x in (50, 80, 20, 300, 1, 33)]
    ql = [1, 0, 3, 0, 1, 2]
    batch = wl.custom_batch(LLAMA, seq, ql, 450, shared_prefix_blocks=shared)
    buf, _ = _run(batch)
    assert plan_record(buf)["cascade_blocks"] == shared
