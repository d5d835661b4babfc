"""Shared parity helpers: run one step through the C ABI and compare it with
the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_attention_kv_gb300 import binding as pkv
from paged_attention_kv_gb300 import workloads as wl

# Attention tolerance against the fp64 oracle on bf16 outputs.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def host_inputs(tensors: dict) -> dict:
    return {k: wl.bf16_bits(v).copy() for k, v in tensors.items()}


def oracle_step(batch, host: dict, rows=None, num_threads=None):
    """Oracle slot mapping, KV write (into a copy of the pool) and attention."""
    slots = oracle.slot_mapping(batch.block_table, batch.seq_lens, batch.query_start_loc, batch.num_blocks)
    pool = host["kv_cache"].copy()
    oracle.kv_write(pool, host["k"], host["v"], slots)
    out = oracle.paged_attention(host["q"], pool, batch.block_table, batch.seq_lens, batch.query_start_loc,
                                 batch.scale, rows=rows, num_threads=num_threads)
    return slots, pool, out


def attention_errors(got_bf16: torch.Tensor, ref: np.ndarray, rows=None):
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        rows = np.asarray(rows)
        got = got[rows[:, 0], rows[:, 1]]
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0, rms, got


def assert_attention_close(got_bf16, ref, rows=None, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what="", rel=0.0):
    """Element-wise |got - ref| <= max_abs + rel * |ref| and mean-abs <= mean_abs.
    rel is 0 for the workloads' bar; peaked inputs whose outputs approach
    single V values (|O| of several units) add the bf16 terms that scale
    with |O|."""
    mx, mn, rms, got = attention_errors(got_bf16, ref, rows)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if rel:
        excess = np.abs(got - ref) - rel * np.abs(ref)
        mx = float(excess.max()) if excess.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3e} mean-abs {mn:.3e} (ref rms {rms:.3e})"
    return mx, mn


def device_tensors(batch, device="cuda", generate_on=None, sentinel=True):
    """Seeded tensors for `batch` on the GPU (drawn on `generate_on`)."""
    gen_dev = generate_on or device
    ten = wl.make_tensors(batch, device=gen_dev, sentinel_unreferenced=sentinel)
    return {k: v.to(device) for k, v in ten.items()}


def run_gpu_step(batch, dev_tensors, workspace_bytes=None):
    """Slot mapping + KV write + attention through the C ABI; returns host
    slot mapping, pool bits, output tensor and the two status words."""
    buf = pkv.StepBuffers(batch, dev_tensors)
    if workspace_bytes is not None:
        buf.workspace = torch.empty((workspace_bytes + 7) // 8, dtype=torch.int64, device=buf.q.device)
    buf.step()
    torch.cuda.synchronize()
    st = pkv.pkv_read_status(buf.status)
    wst = pkv.pkv_read_status(buf.workspace)
    return buf, st, wst
