"""Pins the fp64 oracle to facts fixed outside itself: the pages' worked
numbers (tests/golden), closed forms, a dense textbook attention built a
different way, and invariants the method must have.

Source: "Inside vLLM: Anatomy of a High-Throughput LLM Inference System"
(pages 1-3). Each test names the passage it leans on.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
B = 16


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bf16(x):
    """fp32 -> bf16 bit patterns, round to nearest even."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _f(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _random_case(seed, hq, hkv, d, seq_lens, q_lens, pool_blocks=None, shared=0):
    """A small random batch: block tables from a shuffled pool, N(0,1) bf16."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    nbr = [max(1, -(-int(L) // B)) for L in seq_lens]
    need = shared + sum(n - shared for n in nbr)
    nb = pool_blocks or need + 5
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(nbr), max(nbr)), -1, np.int32)
    cur = shared
    for r, n in enumerate(nbr):
        bt[r, :shared] = perm[:shared]
        bt[r, shared:n] = perm[cur:cur + n - shared]
        cur += n - shared
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    t = int(qsl[-1])
    q = _bf16(rng.standard_normal((t, hq, d)))
    cache = _bf16(rng.standard_normal((nb, 2, hkv, B, d)))
    return q, cache, bt, seq_lens, qsl


# --- pages' worked numbers -------------------------------------------------

def test_block_bytes_matches_page_formula_values():
    """Page 2, "LLM Engine 构造函数": bytes per block per layer."""
    rows = _golden_rows("block_size.txt")
    assert len(rows) == 3
    for name, bs, hkv, d, dt, expect in rows:
        assert oracle.block_bytes(int(bs), int(hkv), int(d), int(dt)) == int(expect), name


@pytest.mark.parametrize("hkv,d,expect", [(4, 64, 16384), (8, 128, 65536)])
def test_cache_layout_block_is_one_contiguous_formula_sized_unit(hkv, d, expect):
    """Filling every slot of one block through the oracle's KV write must
    change exactly the formula's byte count (page 2 block-size note), as
    one contiguous run at block_id * bytes_per_block."""
    nb = 5
    cache = np.zeros((nb, 2, hkv, B, d), np.uint16)
    block = 3
    k = np.full((B, hkv, d), 0x3F81, np.uint16)  # both bytes nonzero
    v = np.full((B, hkv, d), 0x4001, np.uint16)
    slots = np.arange(block * B, block * B + B, dtype=np.int32)
    oracle.kv_write(cache, k, v, slots)
    raw = cache.view(np.uint8).reshape(-1)
    changed = np.nonzero(raw)[0]
    assert changed.size == expect
    assert changed[0] == block * expect and changed[-1] == (block + 1) * expect - 1


def test_blocks_needed_matches_allocate_slots_example():
    """Page 1 "Scheduler", allocate_slots step 1: 17 tokens -> 2 blocks."""
    for tokens, bs, blocks in _golden_rows("allocate_slots.txt"):
        assert oracle.blocks_needed(int(tokens), int(bs)) == int(blocks)


def test_slot_mapping_17_token_prefill_uses_two_blocks():
    """A 17-token prefill over a table [7, 3]: tokens 0..15 fill block 7,
    token 16 is row 0 of block 3 (ceil(17/16) = 2 blocks are touched)."""
    bt = np.array([[7, 3]], np.int32)
    slots = oracle.slot_mapping(bt, [17], [0, 17], num_blocks=8)
    assert list(slots) == list(range(7 * 16, 8 * 16)) + [3 * 16]
    assert len({s // 16 for s in slots}) == 2


def test_slot_mapping_decode_and_chunk_positions():
    """Decode: the one new token sits at position L-1. Chunk of n tokens:
    positions L-n .. L-1 (page 1 "Chunked prefill": the indexing handles it)."""
    bt = np.array([[5, 2, 9], [1, 4, -1]], np.int32)
    # req 0: L = 40, 1 new token -> position 39 -> block 9 row 7
    # req 1: L = 20, 6 new tokens -> positions 14..19 -> block 1 rows 14,15; block 4 rows 0..3
    slots = oracle.slot_mapping(bt, [40, 20], [0, 1, 7], num_blocks=10)
    assert list(slots) == [9 * 16 + 7, 1 * 16 + 14, 1 * 16 + 15, 64, 65, 66, 67]


def test_chunked_prefill_example_equals_one_shot():
    """Page 1 "Chunked prefill": chunks of 8, prompt x-y-z with z of 2 tokens
    takes 3 steps; the indexing makes the chunked run equal the one-shot run."""
    ((chunk, prompt, steps),) = _golden_rows("chunked_prefill.txt")
    chunk, prompt, steps = int(chunk), int(prompt), int(steps)
    rng = np.random.default_rng(7)
    hq, hkv, d = 4, 2, 16
    nb = 4
    bt = np.array([[2, 0]], np.int32)
    k = _bf16(rng.standard_normal((prompt, hkv, d)))
    v = _bf16(rng.standard_normal((prompt, hkv, d)))
    q = _bf16(rng.standard_normal((prompt, hq, d)))
    scale = 1 / math.sqrt(d)

    # one shot: all 18 tokens written, then attended
    cache1 = np.zeros((nb, 2, hkv, B, d), np.uint16)
    s = oracle.slot_mapping(bt, [prompt], [0, prompt], nb)
    oracle.kv_write(cache1, k, v, s)
    one = oracle.paged_attention(q, cache1, bt, [prompt], [0, prompt], scale)

    # chunked: steps of at most `chunk` new tokens
    cache2 = np.zeros((nb, 2, hkv, B, d), np.uint16)
    outs, done, n_steps = [], 0, 0
    while done < prompt:
        n = min(chunk, prompt - done)
        L = done + n
        s = oracle.slot_mapping(bt, [L], [0, n], nb)
        oracle.kv_write(cache2, k[done:L], v[done:L], s)
        outs.append(oracle.paged_attention(q[done:L], cache2, bt, [L], [0, n], scale))
        done, n_steps = L, n_steps + 1
    assert n_steps == steps
    assert np.array_equal(cache1, cache2)
    assert np.max(np.abs(np.concatenate(outs) - one)) <= 1e-12


def test_two_key_row_worked_by_hand():
    """tests/golden/two_key_softmax.txt: a row computed by hand."""
    vals = {name: float(x) for name, x in _golden_rows("two_key_softmax.txt")}
    cache = np.zeros((1, 2, 1, B, 2), np.uint16)
    cache[0, 0, 0, 0] = _bf16([1, 0])
    cache[0, 0, 0, 1] = _bf16([0, 1])
    cache[0, 1, 0, 0] = _bf16([1, 2])
    cache[0, 1, 0, 1] = _bf16([3, 4])
    q = _bf16([[[1, 0]]])
    out = oracle.paged_attention(q, cache, np.array([[0]], np.int32), [2], [0, 1], 1.0)
    assert abs(out[0, 0, 0] - vals["out0"]) <= 1e-15
    assert abs(out[0, 0, 1] - vals["out1"]) <= 1e-15


# --- closed forms ------------------------------------------------------------

def test_single_key_returns_its_value_exactly():
    q, cache, bt, sl, qsl = _random_case(1, 4, 2, 32, [1], [1])
    out = oracle.paged_attention(q, cache, bt, sl, qsl, 0.3)
    for h in range(4):
        assert np.array_equal(out[0, h], _f(cache[bt[0, 0], 1, h // 2, 0]))


def test_equal_keys_give_mean_of_values():
    q, cache, bt, sl, qsl = _random_case(2, 2, 1, 16, [37], [1])
    for j in range(3):
        cache[bt[0, j], 0, 0, :, :] = _bf16(np.linspace(-1, 1, 16))
    out = oracle.paged_attention(q, cache, bt, sl, qsl, 0.125)
    vals = np.concatenate([_f(cache[bt[0, j], 1, 0]) for j in range(3)])[:37]
    for h in range(2):
        assert np.max(np.abs(out[0, h] - vals.mean(axis=0))) <= 1e-12


def test_dominant_key_selects_its_value():
    d = 16
    q, cache, bt, sl, qsl = _random_case(3, 1, 1, d, [50], [1])
    q[:] = _bf16(np.ones((1, 1, d)))
    hot = 29
    blk, row = bt[0, hot // B], hot % B
    cache[bt[0, :4], 0, 0] = _bf16(np.zeros((4, B, d)))
    cache[blk, 0, 0, row] = _bf16(np.full(d, 8.0))  # score 128 * scale
    out = oracle.paged_attention(q, cache, bt, sl, qsl, 1.0)
    assert np.max(np.abs(out[0, 0] - _f(cache[blk, 1, 0, row]))) <= 1e-12


def test_causal_mask_hides_later_keys():
    """Query i of a chunk sees keys 0..L-n+i only (page 1 "Run forward pass",
    step 3: masks keep each query on what it may attend to)."""
    q, cache, bt, sl, qsl = _random_case(4, 2, 1, 16, [30], [5])
    base = oracle.paged_attention(q, cache, bt, sl, qsl, 0.25)
    # change the key/value at position 29 (visible only to the last query)
    blk, row = bt[0, 29 // B], 29 % B
    cache[blk, :, 0, row] = _bf16(np.full((2, 16), 3.0))
    moved = oracle.paged_attention(q, cache, bt, sl, qsl, 0.25)
    assert np.array_equal(base[:4], moved[:4])
    assert np.max(np.abs(base[4] - moved[4])) > 1e-3


# --- dense textbook attention built a different way --------------------------

def _dense_reference(q, cache, bt, seq_lens, qsl, scale, hq, hkv):
    """Concatenate each request's blocks into contiguous K, V (numpy fancy
    indexing) and apply softmax(Q K^T * scale + causal mask) V per head."""
    qf = _f(q)
    out = np.zeros(qf.shape)
    g = hq // hkv
    for r in range(len(seq_lens)):
        L, s0, s1 = int(seq_lens[r]), int(qsl[r]), int(qsl[r + 1])
        n = s1 - s0
        nblk = -(-L // B)
        kd = _f(cache[bt[r, :nblk], 0])           # [nblk][Hkv][B][D]
        vd = _f(cache[bt[r, :nblk], 1])
        kd = kd.transpose(1, 0, 2, 3).reshape(hkv, nblk * B, -1)[:, :L]
        vd = vd.transpose(1, 0, 2, 3).reshape(hkv, nblk * B, -1)[:, :L]
        pos = np.arange(L - n, L)[:, None]
        mask = np.arange(L)[None, :] > pos
        for h in range(hq):
            s = qf[s0:s1, h] @ kd[h // g].T * scale
            s[mask] = -np.inf
            out[s0:s1, h] = softmax(s, axis=1) @ vd[h // g]
    return out


@pytest.mark.parametrize("seed,hq,hkv,d,seq,ql", [
    (10, 4, 2, 16, [17, 40, 5], [1, 1, 5]),
    (11, 8, 2, 8, [33, 16, 48, 1], [9, 16, 1, 1]),
    (12, 6, 3, 32, [64, 70], [20, 3]),
    (13, 4, 4, 16, [23], [23]),
])
def test_matches_dense_brute_force(seed, hq, hkv, d, seq, ql):
    q, cache, bt, sl, qsl = _random_case(seed, hq, hkv, d, seq, ql)
    scale = 1 / math.sqrt(d)
    got = oracle.paged_attention(q, cache, bt, sl, qsl, scale)
    ref = _dense_reference(q, cache, bt, sl, qsl, scale, hq, hkv)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_row_subset_matches_full():
    q, cache, bt, sl, qsl = _random_case(14, 4, 2, 16, [30, 50], [4, 1])
    full = oracle.paged_attention(q, cache, bt, sl, qsl, 0.2)
    rows = np.array([[0, 3], [4, 1], [2, 0]])
    sub = oracle.paged_attention(q, cache, bt, sl, qsl, 0.2, rows=rows)
    for i, (t, h) in enumerate(rows):
        assert np.array_equal(sub[i], full[t, h])


# --- invariants --------------------------------------------------------------

def test_permuting_physical_blocks_is_bitwise_invariant():
    q, cache, bt, sl, qsl = _random_case(20, 4, 2, 16, [70, 33, 90], [1, 3, 1])
    out = oracle.paged_attention(q, cache, bt, sl, qsl, 0.25)
    rng = np.random.default_rng(21)
    perm = rng.permutation(cache.shape[0]).astype(np.int32)
    cache2 = np.empty_like(cache)
    cache2[perm] = cache
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.paged_attention(q, cache2, bt2, sl, qsl, 0.25)
    assert np.array_equal(out, out2)


def test_shared_prefix_blocks_equal_private_copies():
    """Page 1 "Prefix Caching": a cache hit reuses the same physical blocks.
    Attention over shared blocks equals attention over private copies."""
    hq, hkv, d = 4, 2, 16
    q, cache, bt, sl, qsl = _random_case(30, hq, hkv, d, [70, 90], [1, 1], shared=2)
    assert np.array_equal(bt[0, :2], bt[1, :2])
    shared = oracle.paged_attention(q, cache, bt, sl, qsl, 0.25)
    # give request 1 private copies of the two prefix blocks
    nb = cache.shape[0]
    cache2 = np.concatenate([cache, cache[bt[1, :2]]])
    bt2 = bt.copy()
    bt2[1, :2] = [nb, nb + 1]
    private = oracle.paged_attention(q, cache2, bt2, sl, qsl, 0.25)
    assert np.array_equal(shared, private)


def test_requests_with_identical_content_give_identical_rows():
    hq, hkv, d = 4, 2, 16
    q, cache, bt, sl, qsl = _random_case(31, hq, hkv, d, [50, 50], [1, 1], shared=3)
    cache[bt[1, 3]] = cache[bt[0, 3]]   # same suffix block content
    q[1] = q[0]
    out = oracle.paged_attention(q, cache, bt, sl, qsl, 0.25)
    assert np.array_equal(out[0], out[1])


def test_gqa_query_head_reads_kv_head_h_over_g():
    """Query heads 2h, 2h+1 share kv head h when Hq = 2 Hkv."""
    q, cache, bt, sl, qsl = _random_case(40, 4, 2, 8, [20], [1])
    cache[:, 1, 1] = _bf16(np.full((B, 8), 7.0))
    cache[:, 1, 0] = _bf16(np.full((B, 8), -2.0))
    out = oracle.paged_attention(q, cache, bt, sl, qsl, 0.5)
    assert np.max(np.abs(out[0, 0:2] + 2.0)) <= 1e-14
    assert np.max(np.abs(out[0, 2:4] - 7.0)) <= 1e-14


# --- KV write and error handling --------------------------------------------

def test_kv_write_skips_negative_slots_and_keeps_other_bytes():
    rng = np.random.default_rng(50)
    cache = _bf16(rng.standard_normal((6, 2, 2, B, 8)))
    before = cache.copy()
    k = _bf16(rng.standard_normal((3, 2, 8)))
    v = _bf16(rng.standard_normal((3, 2, 8)))
    oracle.kv_write(cache, k, v, np.array([17, -1, 95], np.int32))
    assert np.array_equal(cache[1, 0, :, 1], k[0]) and np.array_equal(cache[1, 1, :, 1], v[0])
    assert np.array_equal(cache[5, 0, :, 15], k[2]) and np.array_equal(cache[5, 1, :, 15], v[2])
    diff = cache != before
    diff[1, :, :, 1] = False
    diff[5, :, :, 15] = False
    assert not diff.any()


def test_oracle_rejects_bad_batches():
    bt = np.array([[0, 1]], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(bt, [20], [0, 21], num_blocks=4)     # more new tokens than context
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(bt, [40], [0, 1], num_blocks=4)      # context beyond the table
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(np.array([[0, 9]], np.int32), [20], [0, 1], num_blocks=4)  # block outside pool
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(np.zeros((2, 2, 1, B, 8), np.uint16), np.zeros((1, 1, 8), np.uint16),
                        np.zeros((1, 1, 8), np.uint16), np.array([40], np.int32))


# --- block transfer (disaggregated prefill/decode) ---------------------------

def test_block_gather_copies_the_formula_sized_contiguous_unit():
    """Page 1 "Disaggregated P/D": KV moves into / out of paged memory by
    block. A gathered block is exactly the contiguous byte range
    [b * block_bytes, (b + 1) * block_bytes) of the pool (page 2 formula)."""
    rng = np.random.default_rng(60)
    hkv, d = 2, 16
    cache = _bf16(rng.standard_normal((9, 2, hkv, B, d)))
    ids = np.array([7, 0, 3, 7], np.int32)
    got = oracle.kv_gather_blocks(cache, ids)
    nbytes = oracle.block_bytes(B, hkv, d, 2)
    raw = cache.view(np.uint8).reshape(-1)
    for i, b in enumerate(ids):
        assert np.array_equal(got[i].view(np.uint8).reshape(-1), raw[b * nbytes:(b + 1) * nbytes])


def test_block_scatter_then_gather_round_trips_and_touches_only_targets():
    rng = np.random.default_rng(61)
    hkv, d = 2, 8
    cache = _bf16(rng.standard_normal((6, 2, hkv, B, d)))
    before = cache.copy()
    staged = _bf16(rng.standard_normal((2, 2, hkv, B, d)))
    oracle.kv_scatter_blocks(staged, np.array([4, 1], np.int32), cache)
    assert np.array_equal(oracle.kv_gather_blocks(cache, np.array([4, 1], np.int32)), staged)
    untouched = [0, 2, 3, 5]
    assert np.array_equal(cache[untouched], before[untouched])
    with pytest.raises(oracle.OracleError):
        oracle.kv_gather_blocks(cache, np.array([6], np.int32))
