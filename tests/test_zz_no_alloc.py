"""The allocation-free attention entry point (paged_attention_static).

Some callers cannot allocate device memory at the point where they run
attention: an engine that has already given nearly all free device memory to
its KV pool, a plugin whose host framework owns the device memory, or a loop
that cannot afford cudaMalloc's implicit synchronisation. This entry point
serves them from a fixed scratch array inside the library. These tests call
it through the C ABI and check it against the fp64 oracle and against
paged_attention (the entry point that takes a caller workspace) with the
tolerance the parity tests use.

The file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_attention_kv_gb300 import binding as pkv
from paged_attention_kv_gb300 import workloads as wl

from parity_utils import assert_attention_close, device_tensors, host_inputs, oracle_step

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def _static_call(buf, batch, out):
    """One call of paged_attention_static into the caller's `out` (allocated
    beforehand, so that the call itself is the only thing that could take
    device memory)."""
    desc = pkv.cache_desc(buf.kv_cache)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = pkv.LIB.paged_attention_static(
        ctypes.c_void_p(buf.q.data_ptr()), buf.num_tokens, batch.shape.num_q_heads,
        ctypes.c_void_p(buf.kv_cache.data_ptr()), ctypes.byref(desc), ctypes.c_void_p(buf.block_table.data_ptr()),
        batch.num_reqs, batch.max_blocks_per_req, ctypes.c_void_p(buf.seq_lens.data_ptr()),
        ctypes.c_void_p(buf.query_start_loc.data_ptr()), ctypes.c_float(batch.scale),
        ctypes.c_void_p(out.data_ptr()), stream)
    assert rc == pkv.PKV_OK, pkv.status_string(rc)
    return out


def _close(a, b):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert float(d.max()) <= MAX_ABS and float(d.mean()) <= MEAN_ABS, (float(d.max()), float(d.mean()))


def test_static_scratch_matches_workspace_entry_point_on_consecutive_calls():
    results = []
    for name in ("llama8b", "mixed"):
        batch = wl.make_batch(name)
        buf = pkv.StepBuffers(batch, wl.make_tensors(batch, device="cuda"))
        ref = buf.step().clone()          # slot mapping, KV write, attention with a workspace
        torch.cuda.synchronize()
        assert pkv.pkv_read_status(buf.workspace) == 0
        first = _static_call(buf, batch, torch.empty_like(buf.q))
        second_out = torch.empty_like(buf.q)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        second = _static_call(buf, batch, second_out)  # the scratch still holds the previous call's contents
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before
        _close(first, ref)
        _close(second, ref)
        assert torch.equal(first.view(torch.int16), second.view(torch.int16))
        results.append(name)
    assert results == ["llama8b", "mixed"]


@pytest.mark.parametrize("workload", ["tiny", "mixed", "prefix"])
def test_static_scratch_against_the_oracle(workload):
    """Element by element against the fp64 oracle (after the step's KV write,
    which the static entry point does not do), on two calls in a row."""
    batch = wl.make_batch(workload)
    ten = device_tensors(batch)
    host = host_inputs(ten)
    _, pool, ref = oracle_step(batch, host)
    buf = pkv.StepBuffers(batch, ten)
    buf.step()                            # slot mapping and KV write (and attention with a workspace)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bf16_bits(buf.kv_cache), pool)
    for call in range(2):
        out = _static_call(buf, batch, torch.empty_like(buf.q))
        torch.cuda.synchronize()
        assert_attention_close(out, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=f"{workload} static call {call}")


def test_static_scratch_rejects_a_batch_beyond_its_size():
    # 4M new tokens at 32 query heads need a work list larger than the 16 MiB
    # array: refused on the host before anything is launched (the pointers
    # below are never dereferenced).
    desc = pkv.CacheDesc(1024, 16, 8, 128)
    vp = ctypes.c_void_p
    rc = pkv.LIB.paged_attention_static(vp(0x10000), 4 << 20, 32, vp(0x20000), ctypes.byref(desc), vp(0x30000),
                                        4, 8, vp(0x40000), vp(0x50000), ctypes.c_float(0.1), vp(0x60000), vp(0))
    assert rc == pkv.PKV_E_WORKSPACE
