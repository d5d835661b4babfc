"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Bars: slot mapping and KV write bit-exact (integer and byte work); attention
within max-abs 2e-2 and mean-abs 2e-3 of the oracle (bf16 output).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_attention_kv_gb300 import binding as pkv
from paged_attention_kv_gb300 import workloads as wl

from parity_utils import (assert_attention_close, device_tensors, host_inputs, oracle_step, run_gpu_step)

pytestmark = pytest.mark.gpu


def _check_full(batch, ten, workspace_bytes=None, max_abs=2e-2, mean_abs=2e-3, rel=0.0):
    host = host_inputs(ten)
    slots, pool, ref = oracle_step(batch, host)
    buf, st, wst = run_gpu_step(batch, ten, workspace_bytes)
    assert st == 0 and wst == 0, (hex(st), hex(wst))
    assert np.array_equal(buf.slot_mapping.cpu().numpy(), slots)
    assert np.array_equal(wl.bf16_bits(buf.kv_cache), pool)
    assert_attention_close(buf.out, ref, max_abs=max_abs, mean_abs=mean_abs, what=batch.workload, rel=rel)
    return buf, ref


@pytest.mark.parametrize("workload", wl.WORKLOADS)
def test_workload_parity_full(workload):
    """All five workloads at full size: every slot, every pool byte, every
    output element against the oracle."""
    batch = wl.make_batch(workload)
    ten = device_tensors(batch)
    _check_full(batch, ten)


def _custom(shape, seq, ql, seed, **kw):
    return wl.custom_batch(shape, seq, ql, seed, **kw)


LLAMA = wl.LLAMA3_8B
TINY = wl.TINYLLAMA


@pytest.mark.parametrize("shape", [TINY, LLAMA], ids=["d64", "d128"])
def test_context_length_edges(shape):
    seq = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 255, 256, 257, 1000, 4097]
    batch = _custom(shape, seq, [1] * len(seq), 101)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


@pytest.mark.parametrize("ql", [[4, 4, 4, 4], [2, 3, 5, 7], [17, 16, 15, 33]])
def test_multi_token_queries(ql):
    """Several new tokens per request (speculative verify, short chunks):
    causal inside the chunk, tiles straddling token boundaries."""
    seq = [40, 300, 17, 1200]
    batch = _custom(LLAMA, seq, ql, 102)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


def test_prefill_chunks_and_fresh_prompts():
    seq = [100, 700, 513, 64, 2000]
    ql = [100, 200, 513, 1, 37]   # fresh prompts (n = L), a mid chunk, a decode
    batch = _custom(LLAMA, seq, ql, 103)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


@pytest.mark.parametrize("hq,hkv,d", [(32, 32, 128), (32, 16, 64), (32, 8, 64), (32, 4, 128), (32, 2, 128),
                                      (32, 1, 64), (12, 4, 128), (20, 4, 64), (48, 8, 128)])
def test_gqa_groups(hq, hkv, d):
    shape = wl.ModelShape(f"h{hq}-{hkv}-{d}", hq, hkv, d)
    seq = [33, 190, 1024, 7]
    ql = [1, 3, 1, 7]
    batch = _custom(shape, seq, ql, 104 + hq + hkv + d)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


def test_requests_without_new_tokens():
    """A request with n = 0 contributes no rows and must not disturb others."""
    seq = [50, 80, 20, 300, 1]
    ql = [1, 0, 20, 0, 1]
    batch = _custom(LLAMA, seq, ql, 105)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


def test_split_and_unsplit_agree():
    """Minimal workspace (no room for split partials: one CTA per tile) and the
    default (split-KV + merge) both match the oracle and each other."""
    batch = _custom(LLAMA, [3000, 5000, 129, 777], [1, 2, 1, 1], 106)
    ten = device_tensors(batch, generate_on="cpu")
    pristine = {k: v.clone() for k, v in ten.items()}
    s = batch.shape
    minimal = pkv.paged_attention_min_workspace_bytes(batch.num_reqs, batch.num_tokens, s.num_q_heads,
                                                      batch.num_blocks, s.num_kv_heads, s.head_size)
    buf_a, ref = _check_full(batch, ten, workspace_bytes=minimal)
    buf_b, _ = _check_full(batch, pristine)
    assert float((buf_a.out.float() - buf_b.out.float()).abs().max()) <= 2e-2


def test_block_permutation_is_bitwise_invariant():
    """Relabelling physical blocks (and permuting the pool to match) gives the
    same output bits: the arithmetic follows logical key order only."""
    batch = _custom(LLAMA, [900, 47, 3000, 16], [1, 5, 1, 1], 107)
    ten = device_tensors(batch, generate_on="cpu")
    buf_a, _, _ = run_gpu_step(batch, {k: v.clone() for k, v in ten.items()})
    rng = np.random.default_rng(5)
    perm = rng.permutation(batch.num_blocks).astype(np.int32)
    batch2 = wl.Batch(**{**batch.__dict__})
    bt = batch.block_table
    batch2.block_table = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    pool2 = torch.empty_like(ten["kv_cache"])
    pool2[torch.from_numpy(perm).long().to(pool2.device)] = ten["kv_cache"]
    ten2 = {**{k: v.clone() for k, v in ten.items()}, "kv_cache": pool2}
    buf_b, st, wst = run_gpu_step(batch2, ten2)
    assert st == 0 and wst == 0
    assert torch.equal(buf_a.out.view(torch.int16), buf_b.out.view(torch.int16))


def test_chunked_prefill_equals_one_shot():
    """A 2048-token prompt run as one chunk, and as four 512-token chunks
    (each step writes its chunk's KV first): same pool bytes, outputs within
    tolerance of each other and of the oracle."""
    L = 2048
    rng = np.random.default_rng(9)
    g = torch.Generator().manual_seed(9)
    shape = LLAMA
    q = torch.randn(L, shape.num_q_heads, shape.head_size, generator=g).to(torch.bfloat16)
    k = torch.randn(L, shape.num_kv_heads, shape.head_size, generator=g).to(torch.bfloat16)
    v = torch.randn(L, shape.num_kv_heads, shape.head_size, generator=g).to(torch.bfloat16)
    nb = 160
    table = rng.permutation(nb)[:L // 16].astype(np.int32)[None, :]
    pool0 = torch.randn(nb, 2, shape.num_kv_heads, 16, shape.head_size, generator=g).to(torch.bfloat16)

    def batch_for(n, Lc):
        return wl.Batch("chunk", shape, np.array([Lc], np.int32), np.array([n], np.int32), table, nb, 0)

    dev = "cuda"
    one = batch_for(L, L)
    b1, st, wst = run_gpu_step(one, {"q": q.to(dev), "k": k.to(dev), "v": v.to(dev), "kv_cache": pool0.to(dev)})
    assert st == 0 and wst == 0
    pool = pool0.to(dev)
    outs = []
    for c in range(4):
        lo, hi = c * 512, (c + 1) * 512
        bc = batch_for(512, hi)
        buf, st, wst = run_gpu_step(bc, {"q": q[lo:hi].to(dev), "k": k[lo:hi].to(dev), "v": v[lo:hi].to(dev),
                                         "kv_cache": pool})
        assert st == 0 and wst == 0
        outs.append(buf.out)
    chunked = torch.cat(outs)
    assert torch.equal(b1.kv_cache.view(torch.int16), pool.view(torch.int16))
    assert float((chunked.float() - b1.out.float()).abs().max()) <= 2e-2
    host = {"q": wl.bf16_bits(q), "k": wl.bf16_bits(k), "v": wl.bf16_bits(v), "kv_cache": wl.bf16_bits(pool0)}
    _, _, ref = oracle_step(one, host)
    assert_attention_close(chunked, ref, what="chunked")
    assert_attention_close(b1.out, ref, what="one-shot")


def test_garbage_outside_context_is_never_used():
    """Every pool slot outside the requests' contexts holds NaN; the outputs
    must stay finite and match the oracle (masked keys contribute nothing)."""
    batch = _custom(LLAMA, [17, 100, 1023, 45], [1, 3, 1, 45], 108)
    ten = device_tensors(batch, generate_on="cpu")
    full_qsl = np.concatenate([[0], np.cumsum(batch.seq_lens)]).astype(np.int32)
    ctx = oracle.slot_mapping(batch.block_table, batch.seq_lens, full_qsl, batch.num_blocks)
    pool = ten["kv_cache"].cpu()
    keep = torch.zeros(batch.num_blocks * 16, dtype=torch.bool)
    keep[torch.from_numpy(ctx).long()] = True
    keep = keep.view(batch.num_blocks, 1, 1, 16, 1).expand_as(pool)
    poisoned = torch.where(keep, pool, torch.full_like(pool, float("nan")))
    ten["kv_cache"] = poisoned.to("cuda")
    _check_full(batch, ten)


def test_peaked_queries():
    """Q scaled by 4: sharper softmax, a stricter check of the max handling."""
    batch = _custom(LLAMA, [513, 2000, 64, 3333], [1, 1, 4, 1], 109)
    ten = device_tensors(batch, generate_on="cpu")
    ten["q"] = (ten["q"].float() * 4).to(torch.bfloat16)
    _check_full(batch, ten)


def test_bad_metadata_raises_status_without_fault():
    """Out-of-range block ids, slots and lengths are skipped by the kernels'
    own bounds checks and reported in the status words."""
    batch = _custom(LLAMA, [40, 70], [1, 1], 110)
    ten = device_tensors(batch, generate_on="cpu")
    bad = wl.Batch(**{**batch.__dict__})
    bad.block_table = batch.block_table.copy()
    bad.block_table[1, 1] = batch.num_blocks + 7          # read by attention only
    buf, st, wst = run_gpu_step(bad, {k: v.clone() for k, v in ten.items()})
    assert wst & pkv.PKV_DEV_BAD_BLOCK
    # KV write with a slot past the pool: skipped, pool untouched.
    pool = ten["kv_cache"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([batch.num_blocks * 16 + 3, -1], dtype=torch.int32, device="cuda")
    pkv.paged_kv_write(ten["k"], ten["v"], slots, pool, status)
    assert pkv.pkv_read_status(status) & pkv.PKV_DEV_BAD_SLOT
    assert torch.equal(pool.view(torch.int16), ten["kv_cache"].view(torch.int16))
    # More new tokens than context.
    worse = wl.Batch(**{**batch.__dict__})
    worse.seq_lens = np.array([40, 1], np.int32)
    worse.query_lens = np.array([1, 2], np.int32)
    ten3 = device_tensors(worse, generate_on="cpu")
    buf, st, wst = run_gpu_step(worse, ten3)
    assert st & pkv.PKV_DEV_BAD_LEN and wst & pkv.PKV_DEV_BAD_LEN


@pytest.mark.parametrize("shape", [TINY, LLAMA], ids=["d64", "d128"])
def test_chunk_tile_bad_block_is_reported_and_zero_filled(shape):
    """A block id past the pool in a chunk-tile request's table (block 8, the
    first of the second key tile): the chunk kernel's copy warps report
    PKV_DEV_BAD_BLOCK and copy zeros in its place; the rows that never see
    that block (tokens 0-127) and the other request still match the oracle."""
    batch = _custom(shape, [512, 300], [512, 1], 112)
    ten = device_tensors(batch, generate_on="cpu")
    _, _, ref = oracle_step(batch, host_inputs(ten))
    bad = wl.Batch(**{**batch.__dict__})
    bad.block_table = batch.block_table.copy()
    bad.block_table[0, 8] = batch.num_blocks + 7
    buf, st, wst = run_gpu_step(bad, {k: v.clone() for k, v in ten.items()})
    assert wst & pkv.PKV_DEV_BAD_BLOCK
    assert torch.isfinite(buf.out.float()).all()
    keep = list(range(128)) + [512]  # request 0's first 128 tokens, request 1's token
    assert_attention_close(buf.out[keep], ref[keep], what="rows without the bad block")


@pytest.mark.parametrize("workload", ["mixed", "tinyllama"])
def test_repeated_steps_give_the_same_bits(workload):
    """Back-to-back steps on the same inputs (the pipelined launches, the
    chunk kernel beside the split-KV kernel, dynamic work claims) leave clean
    status words and bit-identical outputs every time: a race between the
    kernels' roles would show up as a changed bit or a timeout."""
    batch = wl.make_batch(workload)
    buf = pkv.StepBuffers(batch, device_tensors(batch))
    first = buf.step().clone()
    for i in range(400):
        out = buf.step()
        if i % 100 == 99:
            torch.cuda.synchronize()
            assert pkv.pkv_read_status(buf.status) == 0 and pkv.pkv_read_status(buf.workspace) == 0
            assert torch.equal(out.view(torch.int16), first.view(torch.int16)), f"step {i + 1}"


def test_empty_batch_is_a_no_op():
    q = torch.empty(0, 32, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 2, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    qsl = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = pkv.paged_attention(q, pool, bt, sl, qsl, 0.1)
    assert out.numel() == 0


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (32, 4, 64), (32, 32, 128), (32, 2, 64), (32, 1, 128),
                                      (16, 16, 64), (40, 5, 128)])
def test_chunk_tiles_across_gqa_groups(hq, hkv, d):
    """Requests with at least 128 query rows (tokens x GQA group) run as
    128-row tensor-core chunk tiles: ragged last tiles, chunks at an offset,
    fresh prompts, mixed with decode tokens in one batch."""
    shape = wl.ModelShape(f"chunk-h{hq}-{hkv}-{d}", hq, hkv, d)
    g = hq // hkv
    n_big = max(200 // g, 129 // g + 1)
    seq = [n_big, 700 + n_big, 3 * n_big + 5, 300, 64]
    ql = [n_big, n_big, 2 * n_big + 1, 1, 3]
    batch = _custom(shape, seq, ql, 200 + hq + hkv + d)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


@pytest.mark.parametrize("workload", ["mixed", "tinyllama"])
def test_back_to_back_steps_finish_promptly_with_clean_status(workload):
    """Twenty steps queued back to back (launches overlap across calls) end in
    well under a second each, with no pipeline wait running into its time
    limit, and give the same output as a single step."""
    import time
    batch = wl.make_batch(workload)
    buf = pkv.StepBuffers(batch, device_tensors(batch))
    first = buf.step().clone()
    torch.cuda.synchronize()
    t0 = time.time()
    for _ in range(20):
        buf.step()
    torch.cuda.synchronize()
    assert (time.time() - t0) / 20 < 0.05
    assert pkv.pkv_read_status(buf.status) == 0
    assert pkv.pkv_read_status(buf.workspace) == 0
    assert torch.equal(first.view(torch.int16), buf.out.view(torch.int16))


@pytest.mark.parametrize("workload", ["tinyllama", "mixed"])
def test_graph_replay_matches_eager_step(workload):
    """A step captured into a CUDA graph and replayed gives the same bits as
    the eager step, with clean status words."""
    batch = wl.make_batch(workload)
    ten = device_tensors(batch)
    eager = pkv.StepBuffers(batch, {k: v.clone() for k, v in ten.items()})
    ref = eager.step().clone()
    g = pkv.StepGraph(pkv.StepBuffers(batch, ten))
    for _ in range(3):
        out = g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert pkv.pkv_read_status(g.buffers.status) == 0
    assert pkv.pkv_read_status(g.buffers.workspace) == 0


@pytest.mark.parametrize("shape", [TINY, LLAMA], ids=["d64", "d128"])
def test_kv_block_gather_scatter_bit_exact(shape):
    """Block-granular transfer for disaggregated prefill/decode: gather and
    scatter match the oracle byte for byte; a bad id is skipped and flagged."""
    batch = _custom(shape, [300, 1000, 77], [1, 1, 1], 300)
    ten = device_tensors(batch, generate_on="cpu")
    pool = ten["kv_cache"]
    host_pool = wl.bf16_bits(pool).copy()
    rng = np.random.default_rng(301)
    ids = rng.choice(batch.num_blocks, size=37, replace=False).astype(np.int32)
    staged = pkv.paged_kv_gather_blocks(pool, torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    ref = oracle.kv_gather_blocks(host_pool, ids)
    assert np.array_equal(staged.cpu().numpy().view(np.uint16).reshape(ref.shape), ref)
    # inject fresh blocks into other slots
    dst = rng.choice(np.setdiff1d(np.arange(batch.num_blocks), ids), size=37, replace=False).astype(np.int32)
    fresh = wl.bf16_bits(torch.randn(37, *pool.shape[1:]).to(torch.bfloat16))
    pkv.paged_kv_scatter_blocks(torch.from_numpy(fresh.view(np.uint8).reshape(37, -1)).cuda(),
                                torch.from_numpy(dst).cuda(), pool)
    torch.cuda.synchronize()
    oracle.kv_scatter_blocks(fresh, dst, host_pool)
    assert np.array_equal(wl.bf16_bits(pool), host_pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, batch.num_blocks + 3, -1], dtype=torch.int32, device="cuda")
    pkv.paged_kv_gather_blocks(pool, bad, status=status)
    assert pkv.pkv_read_status(status) & pkv.PKV_DEV_BAD_BLOCK


@pytest.mark.parametrize("workload", ["tinyllama", "mixed"])
def test_host_step_pipeline_matches_device_steps(workload):
    """Steps fed from pinned host memory through the double-buffered
    pipeline (copies overlapping the neighbouring steps' kernels) return, in
    host memory, the same bits as the same steps run on device buffers; two
    query sets alternate so a stale buffer would show."""
    batch = wl.make_batch(workload)
    ten = device_tensors(batch)
    q2 = (ten["q"].float() * -0.5).to(torch.bfloat16)
    refs = []
    for q in (ten["q"], q2):
        buf = pkv.StepBuffers(batch, {**{k: v.clone() for k, v in ten.items()}, "q": q})
        refs.append(buf.step().cpu())
    torch.cuda.synchronize()
    s = batch.shape
    pipe = pkv.HostStepPipeline(ten["kv_cache"].clone(), batch.num_reqs, batch.num_tokens,
                                batch.max_blocks_per_req, s.num_q_heads, batch.scale)
    host = {"k": ten["k"].cpu(), "v": ten["v"].cpu(), "block_table": torch.from_numpy(batch.block_table),
            "seq_lens": torch.from_numpy(batch.seq_lens), "query_start_loc": torch.from_numpy(batch.query_start_loc)}
    qs = [ten["q"].cpu(), q2.cpu()]
    outs = [torch.empty(refs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(5)]
    for i in range(5):
        views = pipe.next_inputs()
        views["q"].copy_(qs[i % 2])
        for k, v in host.items():
            views[k].copy_(v)
        pipe.submit(outs[i])
    pipe.synchronize()
    assert pipe.read_status() == (0, 0)
    for i in range(5):
        assert torch.equal(outs[i].view(torch.int16), refs[i % 2].view(torch.int16)), i


@pytest.mark.parametrize("shape", [TINY, LLAMA], ids=["d64", "d128"])
def test_chunk_tiles_with_ragged_key_ranges(shape):
    """Each 128-row chunk tile is one work item with its own key range:
    requests of 1, 3, 5 and 2 tiles whose tiles end inside a 128-key tile,
    at a block boundary and past several key tiles of prior context."""
    g = shape.num_q_heads // shape.num_kv_heads
    t = 128 // g  # tokens per 128-row tile
    ql = [t, 3 * t, 5 * t, 2 * t, 1]
    seq = [t, 3 * t + 700, 5 * t + 45, 2 * t + 128, 900]
    batch = _custom(shape, seq, ql, 600 + g)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


def test_chunk_tiles_with_scores_growing_along_the_context():
    """Keys scaled up along the context (x (1 + p / 48) at position p) make
    each later 128-key tile's row maxima outgrow the earlier ones by far more
    than 2^8, so the chunk kernel's reference max moves mid-row: P is redone
    against the new reference and O rescaled, in some rows of a warp and not
    in others. The outputs approach single V values (|O| up to 4.4; rounding
    the exact answer to bf16 alone is off by up to 0.0126), so the bar adds
    2^-7 |O|: bf16 output rounding (2^-8 relative) plus bf16 rounding of
    the dominant P weights (2^-8 relative on the numerator only)."""
    seq, ql = [728, 300, 64, 1500], [128, 1, 64, 1]
    batch = _custom(LLAMA, seq, ql, 650)
    ten = wl.make_tensors(batch, device="cpu")
    pool, k = ten["kv_cache"].float(), ten["k"].float()
    qsl = batch.query_start_loc
    for r in (0, 2):
        L, n = seq[r], ql[r]
        pos = np.arange(L - n)
        blk = torch.from_numpy(batch.block_table[r][pos // 16].astype(np.int64))
        tok = torch.from_numpy(pos % 16)
        pool[blk, 0, :, tok, :] *= torch.from_numpy(1.0 + pos / 48.0).float()[:, None, None]
        new = np.arange(L - n, L)
        k[int(qsl[r]):int(qsl[r]) + n] *= torch.from_numpy(1.0 + new / 48.0).float()[:, None, None]
    ten["kv_cache"], ten["k"] = pool.to(torch.bfloat16), k.to(torch.bfloat16)
    _check_full(batch, {key: val.to("cuda") for key, val in ten.items()}, rel=2.0 ** -7)


def test_max_query_len_bound_skips_the_chunk_kernel_and_stays_correct():
    """paged_attention_bounded: a decode batch gives the same bits with and
    without the bound (the bound only drops the chunk kernel's launch); a
    bound too small for the batch's chunk requests sends their rows down the
    split-KV path, still within tolerance of the oracle."""
    dec = _custom(LLAMA, [300, 1200, 47, 2000], [1, 1, 1, 1], 660)
    ten = device_tensors(dec, generate_on="cpu")
    buf = pkv.StepBuffers(dec, {k: v.clone() for k, v in ten.items()})
    buf.step()
    with_bound = buf.out.clone()
    pkv.paged_attention(buf.q, buf.kv_cache, buf.block_table, buf.seq_lens, buf.query_start_loc, dec.scale,
                        buf.out, buf.workspace)
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(buf.workspace) == 0
    assert torch.equal(with_bound.view(torch.int16), buf.out.view(torch.int16))

    mixed = _custom(LLAMA, [700, 90, 1500], [200, 1, 64], 661)
    ten = device_tensors(mixed, generate_on="cpu")
    host = host_inputs(ten)
    slots, pool, ref = oracle_step(mixed, host)
    buf = pkv.StepBuffers(mixed, ten)
    buf.max_query_len = 1  # too small: requests 0 and 2 have 800 and 256 rows
    buf.step()
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(buf.status) == 0 and pkv.pkv_read_status(buf.workspace) == 0
    h = buf.workspace[:8].view(torch.int32).cpu().numpy()
    assert int(h[6]) == 0  # no chunk items: every row went to the split-KV path
    assert_attention_close(buf.out, ref, what="too-small bound")


@pytest.mark.parametrize("workload", ["tiny", "mixed"])
def test_prepared_step_matches_the_checked_calls(workload):
    """StepBuffers.prepared(): the same three C calls with prebuilt
    arguments give the same slot mapping, pool and output bits."""
    batch = wl.make_batch(workload)
    ten = device_tensors(batch, generate_on="cpu")
    a = pkv.StepBuffers(batch, {k: v.clone() for k, v in ten.items()})
    b = pkv.StepBuffers(batch, {k: v.clone() for k, v in ten.items()})
    a.step()
    run = b.prepared()
    run()
    torch.cuda.synchronize()
    for buf in (a, b):
        assert pkv.pkv_read_status(buf.status) == 0 and pkv.pkv_read_status(buf.workspace) == 0
    assert torch.equal(a.slot_mapping, b.slot_mapping)
    assert torch.equal(a.kv_cache.view(torch.int16), b.kv_cache.view(torch.int16))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


@pytest.mark.parametrize("hkv,d,tokens", [(3, 72, 37), (5, 80, 130), (1, 8, 300), (8, 128, 1000), (2, 256, 65)],
                         ids=["27-chunk-rows", "50-chunk-rows", "1-chunk-rows", "128-chunk-rows", "64-chunk-rows"])
def test_kv_write_row_widths_bit_exact(hkv, d, tokens):
    """The KV write takes 1, 2 or 4 token rows per warp pass by row width
    (hkv x d / 8 16-byte chunks); rows of every width class, ragged ones
    included, land bit for bit where the oracle puts them, slots of -1 are
    skipped and every other slot keeps its sentinel."""
    rng = np.random.default_rng(hkv * 1000 + d)
    nb = (tokens + 15) // 16 * 2
    slots = rng.permutation(nb * 16)[:tokens].astype(np.int32)
    slots[rng.random(tokens) < 0.1] = -1
    g = torch.Generator().manual_seed(hkv + d)
    k = torch.randn(tokens, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(tokens, hkv, d, generator=g).to(torch.bfloat16)
    pool = torch.full((nb, 2, hkv, 16, d), float("nan"), dtype=torch.bfloat16)
    ref = wl.bf16_bits(pool).copy()
    oracle.kv_write(ref, wl.bf16_bits(k), wl.bf16_bits(v), slots)
    dev_pool = pool.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_write(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), dev_pool, status)
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(status) == 0
    assert np.array_equal(wl.bf16_bits(dev_pool), ref)


def test_fused_slot_mapping_and_kv_write_match_the_two_calls():
    """paged_kv_write_slots gives the slot mapping, pool and status bits of
    paged_slot_mapping followed by paged_kv_write, including a token whose
    block-table entry is out of range (flagged, its K/V skipped)."""
    batch = _custom(LLAMA, [300, 17, 700, 64], [5, 1, 200, 64], 670)
    ten = device_tensors(batch, generate_on="cpu")
    bt = batch.block_table.copy()
    bt[1, 1] = batch.num_blocks + 5  # request 1's new token (position 16) lands in block slot 1
    dev = {k: v.clone() for k, v in ten.items()}
    bt_d = torch.from_numpy(bt).cuda()
    sl_d = torch.from_numpy(batch.seq_lens).cuda()
    qsl_d = torch.from_numpy(batch.query_start_loc).cuda()
    t = batch.num_tokens
    st_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots_a = pkv.paged_slot_mapping(bt_d, sl_d, qsl_d, t, batch.num_blocks, status=st_a)
    pool_a = dev["kv_cache"].clone()
    pkv.paged_kv_write(dev["k"], dev["v"], slots_a, pool_a, st_a)
    st_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots_b = torch.full((t,), 12345, dtype=torch.int32, device="cuda")
    pool_b = dev["kv_cache"].clone()
    desc = pkv.cache_desc(pool_b)
    import ctypes
    vp = ctypes.c_void_p
    rc = pkv.LIB.paged_kv_write_slots(vp(dev["k"].data_ptr()), vp(dev["v"].data_ptr()), vp(bt_d.data_ptr()),
                                      batch.num_reqs, bt.shape[1], vp(sl_d.data_ptr()), vp(qsl_d.data_ptr()), t,
                                      vp(pool_b.data_ptr()), ctypes.byref(desc), vp(slots_b.data_ptr()),
                                      vp(st_b.data_ptr()), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(st_a) == pkv.pkv_read_status(st_b) == pkv.PKV_DEV_BAD_BLOCK
    assert torch.equal(slots_a, slots_b)
    assert int(slots_b[5].item()) == -1
    assert torch.equal(pool_a.view(torch.int16), pool_b.view(torch.int16))


def test_a_wait_that_never_completes_is_reported_and_the_context_survives():
    """Failure detection without a fault: the self-test's wait on a barrier
    that nothing arrives on gives up after 2 ms, the status word carries
    PKV_DEV_TIMEOUT, and the next attention step runs normally."""
    import time
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    pkv.pkv_selftest_bounded_wait(status, timeout_us=2000)
    torch.cuda.synchronize()
    assert time.time() - t0 < 1.0
    assert pkv.pkv_read_status(status) == pkv.PKV_DEV_TIMEOUT
    batch = _custom(LLAMA, [300, 40], [1, 2], 610)
    _check_full(batch, device_tensors(batch, generate_on="cpu"))


def test_duplicate_slots_stay_inside_their_slot():
    """Two tokens mapped to one slot (an invalid slot mapping that the write
    does not detect): every 16-byte chunk of that slot ends up as one of the
    two tokens' chunks, and no other byte of the pool changes."""
    batch = _custom(TINY, [40, 70], [1, 1], 620)
    ten = device_tensors(batch, generate_on="cpu")
    pool = ten["kv_cache"].clone()
    before = wl.bf16_bits(pool).copy()
    k = torch.randn(3, TINY.num_kv_heads, TINY.head_size).to(torch.bfloat16).cuda()
    v = torch.randn(3, TINY.num_kv_heads, TINY.head_size).to(torch.bfloat16).cuda()
    slot = 5 * 16 + 7
    slots = torch.tensor([slot, slot, 9 * 16 + 1], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_write(k, v, slots, pool, status)
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(status) == 0
    after = wl.bf16_bits(pool)
    kb, vb = wl.bf16_bits(k), wl.bf16_bits(v)
    changed = np.argwhere(before != after)
    blocks_rows = {(int(c[0]), int(c[3])) for c in changed}
    assert blocks_rows <= {(5, 7), (9, 1)}
    for kv, src in ((0, kb), (1, vb)):
        got = after[5, kv, :, 7, :].reshape(TINY.num_kv_heads, -1, 8)  # 16-byte chunks
        a0 = src[0].reshape(TINY.num_kv_heads, -1, 8)
        a1 = src[1].reshape(TINY.num_kv_heads, -1, 8)
        ok = np.all(got == a0, axis=2) | np.all(got == a1, axis=2)
        assert ok.all()
        assert np.array_equal(after[9, kv, :, 1, :], src[2])


@pytest.mark.parametrize("case", ["mixed", "chunk_heavy", "chunk_only"])
def test_chunk_kernel_beside_split_kv_gives_the_serial_bits(case):
    """With chunk tiles, the chunk kernel runs beside the split-KV kernel on
    the share of the SMs the work list sets (all of them when the decode part
    is negligible); with timing events the two run one after the other. Both
    orders must give the same bits (each output row is computed by one kernel
    in a fixed order), within tolerance of the oracle, and the share must lie
    in [1, SMs]."""
    if case == "mixed":
        batch = wl.make_batch("mixed")
    elif case == "chunk_heavy":  # long prefill chunks beside a handful of short decodes
        batch = _custom(LLAMA, [4096, 3000, 64, 200, 33], [2048, 1024, 1, 1, 1], 671)
    else:  # no split-KV rows at all
        batch = _custom(TINY, [1024, 700], [512, 256], 672)
    ten = device_tensors(batch, generate_on="cpu")
    host = host_inputs(ten)
    slots, pool, ref = oracle_step(batch, host)
    buf = pkv.StepBuffers(batch, ten)
    buf.step()
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(buf.status) == 0 and pkv.pkv_read_status(buf.workspace) == 0
    beside = buf.out.clone()
    h = buf.workspace[:16].view(torch.int32).cpu().numpy()
    n_chunk_items, chunk_ctas = int(h[6]), int(h[11])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert n_chunk_items > 0
    assert 1 <= chunk_ctas <= sms, chunk_ctas
    if case != "mixed":
        assert chunk_ctas == sms  # the split-KV side is under a microsecond
    assert_attention_close(beside, ref, what=f"{case} beside")

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    buf.out.zero_()
    pkv.paged_attention(buf.q, buf.kv_cache, buf.block_table, buf.seq_lens, buf.query_start_loc, batch.scale,
                        buf.out, buf.workspace, events=ev)
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(buf.workspace) == 0
    assert torch.equal(beside.view(torch.int16), buf.out.view(torch.int16))
