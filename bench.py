#!/usr/bin/env python
"""Benchmark of one paged-KV attention step on GB300.

A step is the whole hot path over one batch: slot mapping, the KV write of
the step's new tokens, and attention (work-list kernel, then the split-KV
attention kernel, which also merges split partials), all through the C ABI. The default
workload is the Llama-3-8B-shaped decode batch (32 q / 8 kv heads, head 128,
256 requests with contexts uniform in [512, 4096], block size 16); its pool
(~3 GB) and per-step KV reads (~2.3 GB) are far larger than the 129 MB L2.

Prints one JSON line. ``value`` is query tokens per second for the whole job
(all ranks) with inputs resident in HBM; ``e2e`` is the same metric with
each step's inputs copied from pinned host memory and the output copied back
inside the timed region. ``roofline`` covers the attention kernel, timed
live with CUDA events on its stream; ``cpu_baseline`` is the fp64 oracle on
the host cores over a bounded sample of the same workload.

``--impl reference`` times the oracle itself (the reference arm of this
comparison) on the same workload and prints the same line shape.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

METRIC = "decode attention tokens/s and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
UNIT = "tokens/s"
KERNEL_SOURCES = ("attention.cu", "attention_plan.cuh", "pkv_device.cuh")
PROFILE_DOC = os.path.join(REPO, "profiles", "attention_decode_kernel_llama8b.md")
KERNEL_SOURCES_CHUNK = ("attention_chunk.cu", "attention_chunk.h", "attention_plan.cuh", "pkv_device.cuh")
PROFILE_DOC_CHUNK = os.path.join(REPO, "profiles", "chunk_kernel_mixed.md")


def launches_per_step(batch) -> int:
    """Kernels one timed step launches (the prepared step): slot mapping with
    the KV write (one launch), the work list, split-KV attention, and the
    chunk-tile kernel when a request's new tokens can fill a 128-row tile
    (the step passes its longest query to the library, which skips the
    launch otherwise)."""
    g = batch.shape.num_q_heads // batch.shape.num_kv_heads
    longest = int(batch.query_lens.max()) if batch.num_reqs else 0
    chunk = 128 % g == 0 and batch.num_tokens * g >= 128 and longest * g >= 128
    return 3 + (1 if chunk else 0)


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="llama8b")
    p.add_argument("--skip-cpu-baseline", action="store_true", help="leave out the oracle CPU baseline")
    p.add_argument("--skip-e2e", action="store_true", help="leave out the end-to-end (host buffers) loop")
    p.add_argument("--graph", action="store_true",
                   help="replay the step from a captured CUDA graph in the timed loop")
    p.add_argument("--l2", choices=("auto", "layers", "flush", "none"), default="auto",
                   help="keeping L2 cold between steps. layers: consecutive steps use distinct KV pools (one "
                        "per model layer, as a real step over a model's layers does) until their total exceeds "
                        "512 MiB; flush: write and read 512 MiB before every step and time steps one by one; "
                        "auto: layers when one pool is under 512 MiB, else none (the step's reads are GBs)")
    p.add_argument("--op", choices=("step", "kv_transfer", "kv_write"), default="step",
                   help="kv_transfer: time block gather + scatter of the workload's context blocks; "
                        "kv_write: time the KV write alone, on the workload's new tokens and on a "
                        "prefill-sized token count")
    return p.parse_args()


# --------------------------------------------------------------------------
# workload bookkeeping (measurement only)
# --------------------------------------------------------------------------

L2_SCRUB_BYTES = 512 << 20


def scrub_l2(scrub) -> None:
    """Evict the step's data from L2: write a buffer four times the L2 size,
    then read all of it back so the lines left behind are clean (no
    write-backs land in the timed step)."""
    import torch
    scrub.zero_()
    scrub.view(torch.int64).sum()


def pool_bytes(batch) -> int:
    s = batch.shape
    return batch.num_blocks * 2 * 16 * s.num_kv_heads * s.head_size * 2


def l2_mode(args, batch) -> tuple[str, int]:
    """('layers', number of distinct pools) | ('flush', 1) | ('none', 1)."""
    mode = args.l2
    if mode == "auto":
        mode = "layers" if pool_bytes(batch) < L2_SCRUB_BYTES else "none"
    if mode == "layers":
        return mode, max(2, -(-L2_SCRUB_BYTES // pool_bytes(batch)))
    return mode, 1


def l2_note(batch, mode: str, layers: int) -> str:
    if mode == "flush":
        return "L2 flushed before every timed step (512 MiB written then read), steps timed one by one"
    if mode == "layers":
        return (f"inputs larger than L2: consecutive steps rotate over {layers} distinct KV pools (one per layer, "
                f"{layers * pool_bytes(batch) / 1e6:.0f} MB in total vs 129 MB L2), no flush")
    return f"inputs larger than L2 (pool of {pool_bytes(batch) / 1e9:.2f} GB vs 129 MB L2), no flush"


def workload_config(batch, l2: str = "") -> dict:
    s = batch.shape
    return {
        "workload": batch.workload,
        "description": batch.description,
        "shape": f"{s.name} attention ({s.num_q_heads} q / {s.num_kv_heads} kv heads, head {s.head_size})",
        "num_reqs": batch.num_reqs,
        "num_tokens": batch.num_tokens,
        "block_size": 16,
        "num_blocks": batch.num_blocks,
        "context_tokens": int(batch.seq_lens.sum()),
        "l2": l2 or l2_note(batch, "none", 1),
    }


def chunk_requests(batch) -> np.ndarray:
    """Requests the chunk-tile kernel takes: >= 128 query rows (new tokens x
    GQA group) when a 128-row tile holds whole tokens."""
    g = batch.shape.num_q_heads // batch.shape.num_kv_heads
    if 128 % g != 0 or batch.num_tokens * g < 128:
        return np.zeros(batch.num_reqs, dtype=bool)
    return batch.query_lens.astype(np.int64) * g >= 128


def chunk_flops(batch) -> float:
    """Causal-exact flops of the chunk tiles: 4 * D per (query row, visible key)."""
    s = batch.shape
    g = s.num_q_heads // s.num_kv_heads
    total = 0
    for r in np.nonzero(chunk_requests(batch))[0]:
        n, L = int(batch.query_lens[r]), int(batch.seq_lens[r])
        visible = np.arange(L - n + 1, L + 1, dtype=np.int64).sum()
        total += 4 * s.head_size * g * s.num_kv_heads * int(visible)
    return float(total)


def algorithmic_bytes(batch, only=None) -> dict:
    """Bytes one attention launch must move at minimum: every context
    token's K and V once (blocks shared by several requests counted once),
    Q read, output written, the block-table entries used and the per-request
    metadata. `only`: a boolean mask of the requests to count (one kernel's
    share)."""
    s = batch.shape
    sel = np.ones(batch.num_reqs, dtype=bool) if only is None else np.asarray(only)
    rows_used = {}
    for r, L in enumerate(batch.seq_lens):
        if not sel[r]:
            continue
        L = int(L)
        nb = -(-L // 16)
        for j in range(nb):
            b = int(batch.block_table[r, j])
            rows = min(16, L - 16 * j)
            if rows_used.get(b, 0) < rows:
                rows_used[b] = rows
    unique_tokens = sum(rows_used.values())
    per_token = 2 * s.num_kv_heads * s.head_size * 2
    kv = unique_tokens * per_token
    logical_kv = int(batch.seq_lens[sel].sum()) * per_token
    qo = 2 * int(batch.query_lens[sel].sum()) * s.num_q_heads * s.head_size * 2
    bt = int(sum(-(-int(L) // 16) for L in batch.seq_lens[sel])) * 4
    meta = (2 * int(sel.sum()) + 1) * 4
    return {"kv": kv, "logical_kv": logical_kv, "q_out": qo, "block_table": bt, "meta": meta,
            "attention_total": kv + qo + bt + meta, "unique_tokens": unique_tokens}


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(REPO, "paged_attention_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(doc=PROFILE_DOC, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        text = open(doc).read()
    except OSError:
        return None
    src = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not src or not val or src.group(1) != kernel_source_hash(sources):
        return None
    return float(val.group(1))


def measured_peaks() -> dict:
    try:
        with open(os.path.join(REPO, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def chunk_roofline(batch, chunk_ms: float, peaks: dict) -> dict:
    """The chunk-tile kernel against the bf16 tensor peak (a contraction)."""
    fl = chunk_flops(batch)
    achieved = fl / (chunk_ms * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": "chunk_kernel (tcgen05)", "achieved": achieved,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "peak_source": f"{peaks['source']} cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
            "flops_per_launch": fl, "kernel_us": chunk_ms * 1e3,
            "traffic": profiled_traffic(PROFILE_DOC_CHUNK, KERNEL_SOURCES_CHUNK) if batch.workload == "mixed" else None}


# --------------------------------------------------------------------------
# ranks (weak scaling: independent batches, no data-path collective)
# --------------------------------------------------------------------------

def rank_batch(workload: str, rank: int):
    """Rank r runs its own batch of the workload's shape, drawn from a seed
    offset by 1000 r."""
    from paged_attention_kv_gb300 import workloads as wl
    return wl.make_batch(workload, seed_offset=1000 * rank)


def max_over_ranks(value: float, dist, device=None) -> float:
    """The slowest rank's time (the job's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Query tokens all ranks processed per second of the slowest rank."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-i",
                 str(gpu_index), "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if len(inside) < 3:
            inside, window = rows, "warmup+timed"
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# --------------------------------------------------------------------------
# oracle (CPU baseline and reference arm)
# --------------------------------------------------------------------------

def sub_batch(batch, reqs):
    from paged_attention_kv_gb300 import workloads as wl
    reqs = np.asarray(reqs)
    return wl.Batch(workload=batch.workload, shape=batch.shape, seq_lens=batch.seq_lens[reqs],
                    query_lens=batch.query_lens[reqs], block_table=batch.block_table[reqs],
                    num_blocks=batch.num_blocks, seed=batch.seed)


def oracle_step(batch, host, reqs, threads):
    """Slot mapping, KV write and attention of the requests `reqs` on the
    host cores; returns the query tokens processed."""
    import oracle
    sb = sub_batch(batch, reqs)
    qsl_full = batch.query_start_loc
    tok = np.concatenate([np.arange(qsl_full[r], qsl_full[r + 1]) for r in reqs])
    slots = oracle.slot_mapping(sb.block_table, sb.seq_lens, sb.query_start_loc, sb.num_blocks)
    oracle.kv_write(host["kv_cache"], host["k"][tok], host["v"][tok], slots)
    oracle.paged_attention(host["q"][tok], host["kv_cache"], sb.block_table, sb.seq_lens, sb.query_start_loc,
                           sb.scale, num_threads=threads)
    return int(sb.num_tokens)


def host_copy(ten):
    from paged_attention_kv_gb300 import workloads as wl
    return {k: wl.bf16_bits(v).copy() for k, v in ten.items()}


def cpu_baseline(batch, host, target_s=10.0, cap_s=30.0) -> dict:
    """The oracle as it stands on every host core, over whole requests of
    the workload, repeated until about target_s of work."""
    threads = os.cpu_count() or 1
    order = np.arange(batch.num_reqs)
    t0 = time.perf_counter()
    tokens = oracle_step(batch, host, order[:4], threads)
    per_req = (time.perf_counter() - t0) / 4
    n = int(min(batch.num_reqs, max(4, target_s / max(per_req, 1e-6))))
    done, reqs_done, start = 0, 0, time.perf_counter()
    i = 0
    while time.perf_counter() - start < target_s and time.perf_counter() - start < cap_s:
        sel = order[(np.arange(n) + i) % batch.num_reqs]
        done += oracle_step(batch, host, sel, threads)
        reqs_done += n
        i += n
    el = time.perf_counter() - start
    return {"value": done / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{reqs_done} requests of the {batch.workload} workload ({done} query tokens, whole "
                      f"step: slot mapping + KV write + attention), fp64, {el:.1f} s"}


def run_reference(args, batch, rank):
    """The reference arm: the oracle timed on the host cores."""
    from paged_attention_kv_gb300 import workloads as wl
    if rank != 0:
        return
    ten = wl.make_tensors(batch, device="cpu")
    host = host_copy(ten)
    threads = os.cpu_count() or 1
    # size each step's sample so warmup + steps stay within ~2 minutes
    t0 = time.perf_counter()
    oracle_step(batch, host, np.arange(2), threads)
    per_req = (time.perf_counter() - t0) / 2
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(min(batch.num_reqs, max(1, budget / max(per_req, 1e-6))))
    reqs = [np.arange(i * n, (i + 1) * n) % batch.num_reqs for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle_step(batch, host, reqs[i], threads)
    start = time.perf_counter()
    tokens = 0
    for i in range(args.steps):
        tokens += oracle_step(batch, host, reqs[args.warmup + i], threads)
    el = time.perf_counter() - start
    value = tokens / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(batch),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n} requests of {batch.workload} per step (whole step, fp64)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    batch = rank_batch(args.workload, rank)

    if args.impl == "reference":
        run_reference(args, batch, rank)
        return

    import torch
    from paged_attention_kv_gb300 import binding as pkv
    from paged_attention_kv_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    ten = wl.make_tensors(batch, device=dev)
    if args.op == "kv_transfer":
        run_kv_transfer(args, batch, ten, pkv, torch, dev, dist, rank, world)
        return
    if args.op == "kv_write":
        run_kv_write(args, batch, ten, pkv, torch, dev, dist, rank, world)
        return
    host = host_copy(ten) if (rank == 0 and world == 1 and not args.skip_cpu_baseline) else None
    mode, layers = l2_mode(args, batch)
    bufs = [pkv.StepBuffers(batch, ten)]
    for _ in range(layers - 1):  # one pool per layer; the step's other inputs are shared
        bufs.append(pkv.StepBuffers(batch, {**ten, "kv_cache": ten["kv_cache"].clone()}))
    buf = bufs[0]
    graphs = [pkv.StepGraph(b) for b in bufs] if args.graph else None
    stream = torch.cuda.current_stream()

    nev = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nev)]

    # the headline pass enqueues each step through prebuilt C arguments
    prepared = [b.prepared() for b in bufs]

    def step(i, timed_kernels=False):
        b = bufs[i % layers]
        if graphs is not None and not timed_kernels:
            graphs[i % layers].replay()
            return
        if not timed_kernels:
            prepared[i % layers]()
            return
        pkv.paged_slot_mapping(b.block_table, b.seq_lens, b.query_start_loc, b.num_tokens,
                               batch.num_blocks, b.slot_mapping, b.status)
        pkv.paged_kv_write(b.k, b.v, b.slot_mapping, b.kv_cache, b.status)
        pkv.paged_attention(b.q, b.kv_cache, b.block_table, b.seq_lens, b.query_start_loc, batch.scale,
                            b.out, b.workspace, events=ev[i] if timed_kernels else None,
                            max_query_len=b.max_query_len)

    scrub = torch.empty(L2_SCRUB_BYTES, dtype=torch.uint8, device=dev) if mode == "flush" else None
    sampler = ClockSampler(local_rank)
    for i in range(max(args.warmup, layers)):
        step(i)
    # create the event handles outside the timed region
    for e4 in ev:
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    if scrub is not None:
        # cold L2 every step: scrub, then time the step alone
        ts = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            scrub_l2(scrub)
            ts[i][0].record(stream)
            step(i)
            ts[i][1].record(stream)
        torch.cuda.synchronize()
        elapsed_ms = float(sum(a.elapsed_time(b) for a, b in ts))
    else:
        t_start.record(stream)
        for i in range(args.steps):
            step(i)
        t_end.record(stream)
        torch.cuda.synchronize()
        elapsed_ms = t_start.elapsed_time(t_end)
    wall1 = time.time()
    # Per-kernel pass: the same K steps with events between the attention
    # launches (an event between two launches stops the next one from
    # starting early, so the headline pass above runs without them).
    for i in range(args.steps):
        if scrub is not None:
            scrub_l2(scrub)
        step(i, timed_kernels=True)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    sampler.stop()
    for b in bufs:
        st = pkv.pkv_read_status(b.status)
        wst = pkv.pkv_read_status(b.workspace)
        if st or wst:
            raise RuntimeError(f"device status bits set: {st:#x} {wst:#x}")
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)

    plan_ms = float(np.mean([e4[0].elapsed_time(e4[1]) for e4 in ev]))
    chunk_ms = float(np.mean([e4[1].elapsed_time(e4[2]) for e4 in ev]))
    attn_ms = [e4[2].elapsed_time(e4[3]) for e4 in ev]
    attn_call_ms = [e4[0].elapsed_time(e4[3]) for e4 in ev]
    kernel_ms = float(np.mean(attn_ms))

    # end to end: inputs from pinned host memory, output back, every step
    e2e = None
    if not args.skip_e2e:
        e2e = run_e2e(args, batch, ten, bufs, pkv, torch, dev, dist, scrub)

    cpu = None
    if host is not None:
        cpu = cpu_baseline(batch, host)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    chunk_mask = chunk_requests(batch)
    ab = algorithmic_bytes(batch, only=~chunk_mask)   # what the split-KV kernel reads and writes
    ab_all = algorithmic_bytes(batch)
    peaks = measured_peaks()
    achieved = ab["attention_total"] / (kernel_ms * 1e-3) / 1e9
    ms_per_step = elapsed_ms / args.steps
    value = job_tokens_per_s(world, batch.num_tokens, ms_per_step)
    clocks = sampler.summary(wall0, wall1)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random block tables)",
        "config": {**workload_config(batch, l2_note(batch, mode, layers)), "parallelism": f"{world} independent replicas" if world > 1
                   else "single GPU", "launch": "CUDA graph replay" if graphs is not None else "eager, PDL launches"},
        "roofline": {"bound": "hbm", "kernel": "attention decode_kernel (split-KV)", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     # the committed capture is of the Llama-3-8B batch: other batches get none
                     "traffic": profiled_traffic() if batch.workload == "llama8b" else None,
                     "algorithmic_bytes_per_launch": ab["attention_total"],
                     "kernel_us": kernel_ms * 1e3, "attention_call_us": float(np.mean(attn_call_ms)) * 1e3,
                     "frac_of_8tbps_nominal": achieved / 8000.0},
        "kernels_us": {"work_list": plan_ms * 1e3, "chunk_tiles": chunk_ms * 1e3, "split_kv": kernel_ms * 1e3},
        "roofline_chunk_tiles": chunk_roofline(batch, chunk_ms, peaks) if chunk_mask.any() else None,
        "gpu_launches": launches_per_step(batch) * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "kv_bytes_per_step": {"unique": ab_all["kv"], "logical": ab_all["logical_kv"]},
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_kv_transfer(args, batch, ten, pkv, torch, dev, dist, rank, world):
    """Block-granular KV transfer (disaggregated prefill/decode): gather
    every context block of the batch into a staging buffer, then scatter it
    back. Bytes: each block read once and written once per direction."""
    ids = np.unique(np.concatenate([batch.block_table[r, :-(-int(L) // 16)]
                                    for r, L in enumerate(batch.seq_lens)])).astype(np.int32)
    ids_d = torch.from_numpy(ids).to(dev)
    pool = ten["kv_cache"]
    staging = pkv.paged_kv_gather_blocks(pool, ids_d)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        pkv.paged_kv_gather_blocks(pool, ids_d, staging, status)
        pkv.paged_kv_scatter_blocks(staging, ids_d, pool, status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), dist, dev) / args.steps
    if pkv.pkv_read_status(status):
        raise RuntimeError("device status bits set")
    if rank != 0:
        return
    nbytes = 2 * 2 * ids.shape[0] * pkv.block_bytes(pool)
    peaks = measured_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "KV block transfer (gather + scatter) GB/s", "value": world * achieved, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes)",
        "data": "synthetic", "config": {**workload_config(batch), "blocks": int(ids.shape[0]),
                                        "bytes_per_step": nbytes},
        "roofline": {"bound": "hbm", "kernel": "block_copy_kernel", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": None},
        "gpu_launches": 2 * args.steps}), flush=True)


KV_WRITE_BIG_TOKENS = 65536


def run_kv_write(args, batch, ten, pkv, torch, dev, dist, rank, world):
    """The KV write alone (the scatter of this step's K/V into the pool
    through the slot mapping). Bytes per call: K and V read (2 T Hkv D 2),
    the same written, and the slot mapping (4 T). Timed on the workload's
    own new tokens (small: L2-resident, launch-bound) and on a prefill-sized
    count, KV_WRITE_BIG_TOKENS tokens into distinct slots of a pool of
    1.25x the blocks they need (seeded permutation), which is HBM-bound."""
    s = batch.shape
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    slots = pkv.paged_slot_mapping(torch.from_numpy(batch.block_table).to(dev),
                                   torch.from_numpy(batch.seq_lens).to(dev),
                                   torch.from_numpy(batch.query_start_loc).to(dev), batch.num_tokens,
                                   batch.num_blocks, status=status)
    T = KV_WRITE_BIG_TOKENS
    nblk = -(-T // 16)
    pool_blocks = nblk * 5 // 4
    gen = torch.Generator(device=dev)
    gen.manual_seed(batch.seed + 7)
    k_big = torch.randn((T, s.num_kv_heads, s.head_size), device=dev, generator=gen).to(torch.bfloat16)
    v_big = torch.randn((T, s.num_kv_heads, s.head_size), device=dev, generator=gen).to(torch.bfloat16)
    pool_big = torch.zeros((pool_blocks, 2, s.num_kv_heads, 16, s.head_size), dtype=torch.bfloat16, device=dev)
    perm = torch.randperm(pool_blocks, device=dev, generator=gen)[:nblk].to(torch.int32)
    tok = torch.arange(T, device=dev, dtype=torch.int32)
    slots_big = (perm[tok // 16] * 16 + tok % 16).to(torch.int32)
    cases = {"step": (ten["k"], ten["v"], slots, ten["kv_cache"]), "prefill": (k_big, v_big, slots_big, pool_big)}
    out = {}
    import ctypes
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for name, (k, v, sl, pool) in cases.items():
        pkv.paged_kv_write(k, v, sl, pool, status)  # the checked call once; the timed loop calls the C ABI directly
        desc = pkv.cache_desc(pool)
        cargs = (ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
                 ctypes.c_int32(k.shape[0]), ctypes.c_void_p(pool.data_ptr()), ctypes.byref(desc),
                 ctypes.c_void_p(status.data_ptr()), stream)
        for _ in range(max(3, args.warmup)):
            pkv.LIB.paged_kv_write(*cargs)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            if pkv.LIB.paged_kv_write(*cargs) != 0:
                raise RuntimeError("paged_kv_write failed")
        b.record()
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b), dist, dev) / args.steps
        t = k.shape[0]
        nbytes = 2 * 2 * t * s.num_kv_heads * s.head_size * 2 + 4 * t
        out[name] = {"tokens": int(t), "bytes": nbytes, "us": ms * 1e3, "gbs": nbytes / (ms * 1e-3) / 1e9}
    if pkv.pkv_read_status(status):
        raise RuntimeError("device status bits set")
    if rank != 0:
        return
    peaks = measured_peaks()
    big = out["prefill"]
    print(json.dumps({
        "metric": "KV write GB/s", "value": world * big["gbs"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": big["us"] / 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes)", "data": "synthetic",
        "config": {**workload_config(batch), "cases": out,
                   "note": "value: the prefill-sized case; the step case is the workload's own new tokens "
                           "(L2-resident, launch-bound)"},
        "roofline": {"bound": "hbm", "kernel": "kv_write_kernel", "achieved": big["gbs"],
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": big["gbs"] / peaks["hbm_gbs"],
                     "traffic": None},
        "gpu_launches": 2 * args.steps}), flush=True)


def run_e2e(args, batch, ten, bufs, pkv, torch, dev, dist, scrub=None):
    """K steps through the library's host-buffer pipeline
    (``binding.HostStepPipeline``): every step copies its inputs (q, k, v
    and the metadata tables) from pinned host memory and its output back to
    pinned host memory, inside the timed region; step i+1's input copies
    overlap step i's kernels and step i's output copy overlaps step i+1's.
    The pool stays resident: it is the layer's KV state, not a per-step
    input; with several pools (``bufs``, one per layer) consecutive steps
    rotate over them as in the device-resident pass. With ``scrub`` every
    step runs alone after an L2 flush, copies included."""
    buf = bufs[0]
    layers = len(bufs)
    s = batch.shape
    pipe = pkv.HostStepPipeline(buf.kv_cache, batch.num_reqs, batch.num_tokens, batch.max_blocks_per_req,
                                s.num_q_heads, batch.scale)
    src = {"q": ten["q"].cpu(), "k": ten["k"].cpu(), "v": ten["v"].cpu(), "block_table": buf.block_table.cpu(),
           "seq_lens": buf.seq_lens.cpu(), "query_start_loc": buf.query_start_loc.cpu()}
    for slot in range(pipe.depth):  # the host producer's side: inputs written into each pinned slot once
        views = pipe.slot_inputs(slot)
        for k, v in src.items():
            views[k].copy_(v)
    outs = [torch.empty(buf.out.shape, dtype=buf.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = pipe.packed_bytes
    d2h = outs[0].numel() * outs[0].element_size()

    def submit(i):
        pipe.next_inputs()
        return pipe.submit(outs[i % 2], kv_cache=bufs[i % layers].kv_cache)

    for i in range(max(3, args.warmup)):
        submit(i)
    pipe.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if scrub is not None:
        ms = 0.0
        for i in range(args.steps):
            scrub_l2(scrub)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(pipe.h2d)
            submit(i)
            b.record(pipe.d2h)
            pipe.synchronize()
            ms += a.elapsed_time(b)
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(pipe.h2d)
        for i in range(args.steps):
            submit(i)
        b.record(pipe.d2h)
        pipe.synchronize()
        ms = a.elapsed_time(b)
    st, wst = pipe.read_status()
    if st or wst:
        raise RuntimeError(f"device status bits set in the host-buffer steps: {st:#x} {wst:#x}")
    # the host copy of the output is the device step's output, bit for bit
    last = args.steps - 1
    if not torch.equal(outs[last % 2].view(torch.int16), bufs[last % layers].out.cpu().view(torch.int16)):
        raise RuntimeError("host-buffer step output differs from the device step")
    ms = max_over_ranks(ms, dist, dev)
    world = dist.get_world_size() if dist else 1
    return {"value": job_tokens_per_s(world, batch.num_tokens, ms / args.steps), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps,
            "path": "binding.HostStepPipeline: one packed pinned-host-to-device copy of the step's inputs and one "
                    "device-to-host copy of its output per step, overlapped with the neighbouring steps' kernels"}


if __name__ == "__main__":
    main()
