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
inside the timed region (the median of several timed runs of the K steps).
``roofline`` covers the attention kernel, timed live with CUDA events on its
stream; ``cpu_baseline`` is the fp64 oracle on the host cores over a bounded
sample of the same workload, with a one-thread figure beside it.

After the headline (Llama-3-8B decode) workload the same run times the
prefix-sharing batch and the mixed chunked-prefill + decode batch the same
way and reports them under ``gates``, each with its own roofline(s), per-step
spread and clocks. Clocks are read through NVML every millisecond from a
background thread while the GPU works.

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
    p.add_argument("--gates", default="auto",
                   help="other workloads timed in the same run after the headline one, comma-separated; "
                        "auto: prefix and mixed (the prefix-sharing and mixed batches) when the headline "
                        "workload is llama8b; none: only the headline workload")
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
# NVML clock-event reason bits that the line reports by name.
NVML_REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
                (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))


class NvmlClockSampler:
    """SM clock, power, utilisation and clock-event reasons of one GPU,
    read through NVML (read-only queries of libnvidia-ml) every `interval_s`
    from a background thread, so that even a timed region of a few
    milliseconds holds several samples. Each sample is (wall time, SM MHz,
    max SM MHz, watts, reason bits, GPU utilisation %)."""

    def __init__(self, torch_device_index: int, interval_s: float = 0.001):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if not self._handle_by_uuid(torch_device_index) and \
                self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(torch_device_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.rows = []
        self.interval = interval_s
        self._stop = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _handle_by_uuid(self, idx: int) -> bool:
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(idx).uuid)
        except Exception:
            return False
        name = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        return self.lib.nvmlDeviceGetHandleByUUID(name.encode(), self.ct.byref(self.h)) == 0

    def _run(self):
        ct, lib, h = self.ct, self.lib, self.h

        class Util(ct.Structure):
            _fields_ = [("gpu", ct.c_uint), ("memory", ct.c_uint)]
        clk, pw, rs, ut = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0), Util()
        while not self._stop.is_set():
            t = time.time()
            lib.nvmlDeviceGetClockInfo(h, ct.c_int(1), ct.byref(clk))
            lib.nvmlDeviceGetPowerUsage(h, ct.byref(pw))
            self.reasons_fn(h, ct.byref(rs))
            lib.nvmlDeviceGetUtilizationRates(h, ct.byref(ut))
            self.rows.append((t, float(clk.value), self.max_mhz, pw.value / 1000.0, int(rs.value), int(ut.gpu)))
            self._stop.wait(self.interval)

    def stop(self):
        self._stop.set()
        self.thread.join(timeout=5)


class SmiClockSampler:
    """The same samples from `nvidia-smi --query-gpu ... -lms 20` (used when
    NVML cannot be loaded)."""

    def __init__(self, gpu_index: int):
        self.proc = None
        self.rows = []
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
        bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20, "sw_power_cap": 0x4}
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rb = 0
                for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                   parts[6:10]):
                    if v.lower() == "active":
                        rb |= bits[name]
                self.rows.append((ts + frac, float(parts[2]), float(parts[3]), float(parts[4] or 0), rb, 100))
            except (ValueError, IndexError):
                continue


def start_clock_sampler(local_rank: int):
    try:
        return NvmlClockSampler(local_rank)
    except (OSError, AttributeError):
        return SmiClockSampler(local_rank)


def clock_summary(rows, window, busy, ms_per_step=None) -> dict:
    """Clocks over the timed window (t0, t1); when it holds fewer than three
    samples, over the workload's busy window (its timed, per-kernel and
    per-step passes back to back), and failing that over every sample."""
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    inside = [r for r in rows if window[0] <= r[0] <= window[1]]
    window = "timed"
    if len(inside) < 3:
        inside, window = [r for r in rows if busy[0] <= r[0] <= busy[1]], "this workload's timed and per-kernel passes"
    if len(inside) < 3:
        inside, window = rows, "all samples from warm-up to the last pass"
    reasons = sorted({name for r in inside for bit, name in NVML_REASONS if r[4] & bit})
    mhz = float(np.median([r[1] for r in inside]))
    out = {"sm_mhz": mhz, "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons, "samples": len(inside),
           "window": window, "power_w_max": max(r[3] for r in inside)}
    if ms_per_step is not None:
        out["step_kcycles_at_median_mhz"] = ms_per_step * 1e-3 * mhz * 1e6 / 1e3
    return out


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


def cpu_baseline(batch, host, target_s=10.0, cap_s=30.0, single_s=3.0) -> dict:
    """The oracle as it stands on every host core, over whole requests of
    the workload, repeated until about target_s of work; then the same on one
    thread for about single_s."""
    threads = os.cpu_count() or 1
    order = np.arange(batch.num_reqs)
    t0 = time.perf_counter()
    oracle_step(batch, host, order[:4], threads)
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
    # one thread, whole requests, bounded to about single_s
    done1, reqs1, i, start1 = 0, 0, 0, time.perf_counter()
    while time.perf_counter() - start1 < single_s:
        sel = order[(np.arange(1) + i) % batch.num_reqs]
        done1 += oracle_step(batch, host, sel, 1)
        reqs1 += 1
        i += 1
    el1 = time.perf_counter() - start1
    return {"value": done / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{reqs_done} requests of the {batch.workload} workload ({done} query tokens, whole "
                      f"step: slot mapping + KV write + attention), fp64, {el:.1f} s",
            "single_thread": {"value": done1 / el1, "unit": UNIT, "cores": 1,
                              "sample": f"{reqs1} requests one at a time ({done1} query tokens), fp64, {el1:.1f} s"}}


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

GATE_WORKLOADS = ("prefix", "mixed")


def device_pass(args, batch, ten, pkv, torch, dev, dist, graph=False):
    """One workload with inputs resident in HBM: W warm-up steps, the K
    timed steps back to back (the headline), the same K steps with events
    between the attention launches (per-kernel times) and K steps each
    between two events (the per-step spread)."""
    mode, layers = l2_mode(args, batch)
    bufs = [pkv.StepBuffers(batch, ten)]
    for _ in range(layers - 1):  # one pool per layer; the step's other inputs are shared
        bufs.append(pkv.StepBuffers(batch, {**ten, "kv_cache": ten["kv_cache"].clone()}))
    graphs = [pkv.StepGraph(b) for b in bufs] if graph else None
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    prepared = [b.prepared() for b in bufs]  # the headline pass enqueues each step through prebuilt C arguments

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
                            b.out, b.workspace, events=ev[i], max_query_len=b.max_query_len)

    scrub = torch.empty(L2_SCRUB_BYTES, dtype=torch.uint8, device=dev) if mode == "flush" else None
    for i in range(max(args.warmup, layers)):
        step(i)
    per_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    for e4 in ev:  # create the event handles outside the timed region
        for e in e4:
            e.record(stream)
    for a, b in per_step:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    if scrub is not None:
        # cold L2 every step: scrub, then time the step alone
        for i in range(args.steps):
            scrub_l2(scrub)
            per_step[i][0].record(stream)
            step(i)
            per_step[i][1].record(stream)
        torch.cuda.synchronize()
        step_ms = [x.elapsed_time(y) for x, y in per_step]
        elapsed_ms = float(sum(step_ms))
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
    if scrub is None:
        # Per-step pass: each step between two events (which also stop
        # consecutive steps from overlapping), for the spread of step times.
        for i in range(args.steps):
            per_step[i][0].record(stream)
            step(i)
            per_step[i][1].record(stream)
        torch.cuda.synchronize()
        step_ms = [x.elapsed_time(y) for x, y in per_step]
    wall2 = time.time()
    if dist:
        dist.barrier()
    for b in bufs:
        st = pkv.pkv_read_status(b.status)
        wst = pkv.pkv_read_status(b.workspace)
        if st or wst:
            raise RuntimeError(f"device status bits set ({batch.workload}): {st:#x} {wst:#x}")
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    return {"elapsed_ms": elapsed_ms, "mode": mode, "layers": layers, "bufs": bufs, "scrub": scrub,
            "plan_ms": float(np.mean([e4[0].elapsed_time(e4[1]) for e4 in ev])),
            "chunk_ms": float(np.mean([e4[1].elapsed_time(e4[2]) for e4 in ev])),
            "attn_ms": [e4[2].elapsed_time(e4[3]) for e4 in ev],
            "attn_call_ms": [e4[0].elapsed_time(e4[3]) for e4 in ev],
            "step_ms": step_ms, "window": (wall0, wall1), "busy": (wall0, wall2),
            "graph": graphs is not None}


def spread(ms: list) -> dict:
    a = np.asarray(ms, dtype=np.float64)
    return {"median_ms": float(np.median(a)), "min_ms": float(a.min()), "max_ms": float(a.max()),
            "mean_ms": float(a.mean()), "n": int(a.size)}


def device_fields(batch, res, world, steps, peaks) -> dict:
    """The bench line's device-resident fields of one workload: the headline
    rate, the split-KV kernel's HBM roofline (bytes counted once per
    physical block: a shared prefix counts once), the chunk-tile kernel's
    tensor roofline when the batch has chunk tiles, per-kernel times and the
    per-step spread."""
    chunk_mask = chunk_requests(batch)
    ab = algorithmic_bytes(batch, only=~chunk_mask)  # what the split-KV kernel reads and writes
    ab_all = algorithmic_bytes(batch)
    kernel_ms = float(np.mean(res["attn_ms"]))
    achieved = ab["attention_total"] / (kernel_ms * 1e-3) / 1e9
    ms_per_step = res["elapsed_ms"] / steps
    per_step = spread(res["step_ms"])
    per_step["how"] = ("each step between two CUDA events (no overlap with its neighbours)" if res["mode"] != "flush"
                       else "each step alone after an L2 flush")
    return {
        "value": job_tokens_per_s(world, batch.num_tokens, ms_per_step),
        "ms_per_step": ms_per_step,
        "roofline": {"bound": "hbm", "kernel": "attention decode_kernel (split-KV)", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     # the committed capture is of the Llama-3-8B batch: other batches get none
                     "traffic": profiled_traffic() if batch.workload == "llama8b" else None,
                     "algorithmic_bytes_per_launch": ab["attention_total"],
                     "kernel_us": kernel_ms * 1e3,
                     "kernel_us_spread": {k[:-3] + "_us": v * 1e3 for k, v in spread(res["attn_ms"]).items()
                                          if k.endswith("_ms")},
                     "attention_call_us": float(np.mean(res["attn_call_ms"])) * 1e3,
                     "frac_of_8tbps_nominal": achieved / 8000.0},
        "kernels_us": {"work_list": res["plan_ms"] * 1e3, "chunk_tiles": res["chunk_ms"] * 1e3,
                       "split_kv": kernel_ms * 1e3},
        "roofline_chunk_tiles": chunk_roofline(batch, res["chunk_ms"], peaks) if chunk_mask.any() else None,
        "step_spread": per_step,
        "kv_bytes_per_step": {"unique": ab_all["kv"], "logical": ab_all["logical_kv"]},
    }


def run_gates(args, pkv, torch, wl, dev, dist, rank, world, peaks):
    """The other two configurations the bandwidth target is read on, timed
    the same way in the same run: the prefix-sharing batch (its fraction is
    on unique bytes: the 64 shared blocks count once) and the mixed batch
    (chunk tiles beside split-KV decode: two rooflines)."""
    if args.gates == "auto":
        names = GATE_WORKLOADS if args.workload == "llama8b" else ()
    else:
        names = tuple(x for x in args.gates.split(",") if x)
    out = {}
    for name in names:
        if name == args.workload or name == "none":
            continue
        batch = rank_batch(name, rank)
        ten = wl.make_tensors(batch, device=dev)
        res = device_pass(args, batch, ten, pkv, torch, dev, dist)
        f = device_fields(batch, res, world, args.steps, peaks)
        f["config"] = workload_config(batch, l2_note(batch, res["mode"], res["layers"]))
        f["clocks"] = (res["window"], res["busy"])  # replaced by the summary once the sampler has stopped
        f["gpu_launches"] = launches_per_step(batch) * args.steps
        out[name] = f
        del res, ten
        torch.cuda.empty_cache()
    return out


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
    peaks = measured_peaks()
    sampler = start_clock_sampler(local_rank)
    res = device_pass(args, batch, ten, pkv, torch, dev, dist, graph=args.graph)

    # end to end: inputs from pinned host memory, output back, every step
    e2e = None
    if not args.skip_e2e:
        e2e = run_e2e(args, batch, ten, res["bufs"], pkv, torch, dev, dist, res["scrub"])

    gates = {}
    if args.op == "step" and args.gates != "none":
        del res["bufs"]
        gates = run_gates(args, pkv, torch, wl, dev, dist, rank, world, peaks)
    sampler.stop()

    cpu = None
    if host is not None:
        cpu = cpu_baseline(batch, host)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    fields = device_fields(batch, res, world, args.steps, peaks)
    clocks = clock_summary(sampler.rows, res["window"], res["busy"], fields["ms_per_step"])
    for g in gates.values():
        g["clocks"] = clock_summary(sampler.rows, *g["clocks"], g["ms_per_step"])
    line = {
        "metric": METRIC, "value": fields["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": fields["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random block tables)",
        "config": {**workload_config(batch, l2_note(batch, res["mode"], res["layers"])),
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
                   "launch": "CUDA graph replay" if res["graph"] else "eager, PDL launches"},
        "roofline": fields["roofline"],
        "kernels_us": fields["kernels_us"],
        "roofline_chunk_tiles": fields["roofline_chunk_tiles"],
        "step_spread": fields["step_spread"],
        "gpu_launches": launches_per_step(batch) * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "kv_bytes_per_step": fields["kv_bytes_per_step"],
    }
    if gates:
        line["gates"] = gates
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


E2E_REPS = 5


def run_e2e(args, batch, ten, bufs, pkv, torch, dev, dist, scrub=None):
    """K steps through the library's host-buffer pipeline
    (``binding.HostStepPipeline``): every step copies its inputs (q, k, v
    and the metadata tables) from pinned host memory and its output back to
    pinned host memory, inside the timed region; step i+1's input copies
    overlap step i's kernels and step i's output copy overlaps step i+1's.
    The pool stays resident: it is the layer's KV state, not a per-step
    input; with several pools (``bufs``, one per layer) consecutive steps
    rotate over them as in the device-resident pass. With ``scrub`` every
    step runs alone after an L2 flush, copies included.

    The K steps are timed E2E_REPS times; ``value`` is the median repetition
    (every step of this loop waits on the host for its input slot, so a
    stall of the host thread lands in the timed region; the repetitions
    show whether one did)."""
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
    reps = []
    for _ in range(E2E_REPS):
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
        reps.append(max_over_ranks(ms, dist, dev) / args.steps)
    st, wst = pipe.read_status()
    if st or wst:
        raise RuntimeError(f"device status bits set in the host-buffer steps: {st:#x} {wst:#x}")
    # the host copy of the output is the device step's output, bit for bit
    last = args.steps - 1
    if not torch.equal(outs[last % 2].view(torch.int16), bufs[last % layers].out.cpu().view(torch.int16)):
        raise RuntimeError("host-buffer step output differs from the device step")
    ms_step = float(np.median(reps))
    world = dist.get_world_size() if dist else 1
    return {"value": job_tokens_per_s(world, batch.num_tokens, ms_step), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_step,
            "reps_ms_per_step": reps,
            "how": f"median of {E2E_REPS} timed runs of the same {args.steps} steps",
            "path": "binding.HostStepPipeline: one packed pinned-host-to-device copy of the step's inputs and one "
                    "device-to-host copy of its output per step, overlapped with the neighbouring steps' kernels"}


if __name__ == "__main__":
    main()
