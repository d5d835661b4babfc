"""The seeded generator produces the five workloads' structure."""
import math

import numpy as np
import pytest

from paged_attention_kv_gb300 import workloads as wl


def _blocks(L):
    return -(-int(L) // 16)


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_tables_are_disjoint_pool_prefixes(name):
    b = wl.make_batch(name)
    shared = b.shared_prefix_blocks
    seen = set()
    for r in range(b.num_reqs):
        nb = _blocks(b.seq_lens[r])
        row = b.block_table[r]
        assert (row[:nb] >= 0).all() and (row[:nb] < b.num_blocks).all()
        assert (row[nb:] == -1).all()
        own = row[shared:nb].tolist()
        assert not seen.intersection(own)
        seen.update(own)
    if name != "tiny":
        need = shared + sum(_blocks(L) - shared for L in b.seq_lens)
        assert b.num_blocks == math.ceil(1.25 * need)
    assert b.query_start_loc[-1] == b.num_tokens
    assert (b.query_lens <= b.seq_lens).all()


def test_workload_shapes():
    t = wl.make_batch("tiny")
    assert list(t.seq_lens) == [17, 40] and t.num_blocks == 64 and t.shape.head_size == 64
    tl = wl.make_batch("tinyllama")
    assert tl.num_reqs == 64 and tl.seq_lens.min() >= 128 and tl.seq_lens.max() <= 2048
    l8 = wl.make_batch("llama8b")
    assert l8.num_reqs == 256 and l8.seq_lens.min() >= 512 and l8.seq_lens.max() <= 4096
    mx = wl.make_batch("mixed")
    assert mx.num_tokens == 4 * 512 + 192
    pre = mx.query_lens == 512
    assert sorted(mx.seq_lens[pre].tolist()) == [512, 1024, 1536, 2048]
    dec = ~pre
    assert dec.sum() == 192 and (mx.query_lens[dec] == 1).all()
    assert mx.seq_lens[dec].min() >= 256 and mx.seq_lens[dec].max() <= 4096
    px = wl.make_batch("prefix")
    assert px.num_reqs == 128 and px.shared_prefix_blocks == 64
    assert (px.block_table[:, :64] == px.block_table[0, :64]).all()
    s = px.seq_lens - 1024
    assert s.min() >= 64 and s.max() <= 31744 and px.seq_lens.max() <= 32768
    sd = wl.make_batch("specdec")
    assert sd.num_reqs == 256 and (sd.query_lens == 4).all() and sd.num_tokens == 1024


def test_seeds_are_reproducible_and_distinct():
    a, b = wl.make_batch("llama8b"), wl.make_batch("llama8b")
    assert np.array_equal(a.seq_lens, b.seq_lens) and np.array_equal(a.block_table, b.block_table)
    c = wl.make_batch("llama8b", seed_offset=1000)
    assert not np.array_equal(a.seq_lens, c.seq_lens)


def test_tensors_are_seeded_and_sentinel_marks_unreferenced_blocks():
    b = wl.make_batch("tiny")
    t1 = wl.make_tensors(b)
    t2 = wl.make_tensors(b)
    for k in t1:
        assert np.array_equal(wl.bf16_bits(t1[k]), wl.bf16_bits(t2[k]))
    pool = wl.bf16_bits(t1["kv_cache"])
    used = set(b.block_table[b.block_table >= 0].tolist())
    for blk in range(b.num_blocks):
        is_sentinel = (pool[blk] == wl.SENTINEL_BITS).all()
        assert is_sentinel == (blk not in used)
