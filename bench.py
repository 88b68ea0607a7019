#!/usr/bin/env python3
"""Benchmark of the NVFP4 sparse-MLA decode hot path on GB300.

One step = one pass of the whole path over one batch: quantize-and-append the batch's new
KV tokens (one per query row) into the paged NVFP4 pool, then sparse MLA decode of every
query row (gather, dequant, QK^T, online softmax, PV, split merge).

Workload (N=1 line): B=32 decode rows, s_q=1, h_q=128, topk=2048, 352-B records, a paged pool
of 2,097,152 slots (32,768 pages of 64 tokens, 738 MB), each sequence 65,536 tokens long.
Eight independent index/query sets rotate between steps, so one lap gathers ~185 MB of
distinct records -- more than the 126 MB L2 -- and every step reads its records from HBM.

Prints one JSON line (rank 0). Multi-GPU (torchrun, N ranks): each rank runs its own replica
on its own batch (query rows shard with no exchange), value = rows of all ranks / max time.
`--impl reference` times the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import functools
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "NVFP4 sparse-MLA decode query-tokens/s and % roofline (h_q128,topk2048, 1×GB300)"
UNIT = "query-tokens/s"
N_SETS = 8
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one decode_pair_kernel launch on this workload, from an ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the hash of the decode code
# (comments removed) it was taken with; reported as null once that code changes.
NCU_TRAFFIC = {"f7a55f8541dd": 34268672 + 47104}
DECODE_CALLS_TIMED = 128   # the decode call alone: 16 laps of 8 back-to-back calls


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def code_hash(text: str) -> str:
    """Hash of a C++ source with its // comments and blank lines removed, so that counters
    taken with a kernel stay attached to it across comment-only edits."""
    lines = []
    for line in text.splitlines():
        cut = line.find("//")
        if cut >= 0 and line.count('"', 0, cut) % 2 == 0:
            line = line[:cut]
        line = line.rstrip()
        if line:
            lines.append(line)
    return hashlib.sha1("\n".join(lines).encode()).hexdigest()[:12]


def decode_source_hash() -> str:
    src = os.path.join(ROOT, "nvfp4_kv_cache_sparse_gb300", "csrc", "sparse_decode_pair.cu")
    return code_hash(open(src).read())





# ---------------------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank sets the job time)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(rows_per_rank: int, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank processes its own rows; the job takes the slowest rank's time."""
    return rows_per_rank * world / max_seconds


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons sampled every millisecond during the timed region,
    read through NVML (the library behind nvidia-smi); falls back to `nvidia-smi -lms 100`."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []
        self.max_mhz = None
        self.source = None
        self._stop = None
        self._thread = None
        self._proc = None

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        bus = None
        try:
            p = torch.cuda.get_device_properties(self.cuda_index)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        except AttributeError:
            pass
        if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(handle)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(handle)) != 0:
                raise OSError("no NVML handle")
        return nv, handle

    def __enter__(self):
        import ctypes
        import threading
        try:
            nv, handle = self._nvml_handle()
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._stop = threading.Event()

            def poll():
                clk = ctypes.c_uint()
                rs = ctypes.c_ulonglong()
                while not self._stop.is_set():
                    if nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0:
                        get_reasons(handle, ctypes.byref(rs))
                        self.samples.append((float(clk.value), int(rs.value)))
                    time.sleep(0.001)

            self._thread = threading.Thread(target=poll, daemon=True)
            self._thread.start()
            self.source = "nvml, 1 ms"
        except (OSError, AttributeError):
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.cuda_index), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi, 100 ms"
            except OSError:
                self._proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(f[0]), int(f[2], 16)))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source}
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": self.source}


# ---------------------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------------------

def roofline_numbers(w: synth.DecodeWorkload):
    rows = w.n_rows
    flops = 2.0 * w.h_q * w.topk * (576 + 512) * rows
    bytes_ = rows * (w.topk * w.record_bytes + w.h_q * 576 * 2 + w.topk * 4)
    return flops, bytes_


def roofline_numbers_valid_only(w: synth.DecodeWorkload):
    """The same counting only the used top-k entries (index >= 0): their records and their share
    of the contractions (the index list is still read whole)."""
    used = int((w.indices >= 0).sum())
    flops = 2.0 * w.h_q * used * (576 + 512)
    bytes_ = used * w.record_bytes + w.n_rows * (w.h_q * 576 * 2 + w.topk * 4)
    return flops, bytes_


def pack_layout(parts):
    """Byte offsets of `parts` ((shape, dtype) pairs) laid out one after another in one uint8
    buffer, each starting on a 256-byte boundary, and the buffer's size."""
    offs, n = [], 0
    for shape, dtype in parts:
        offs.append(n)
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        n += -(-nbytes // 256) * 256
    return offs, n


def pack_views(buf: torch.Tensor, parts, offs):
    """Typed, shaped views of a uint8 buffer at the offsets pack_layout gave."""
    return [buf[o:o + int(np.prod(sh)) * torch.empty((), dtype=dt).element_size()].view(dt).view(sh)
            for (sh, dt), o in zip(parts, offs)]


def make_sets(seed: int):
    """N_SETS decode batches over one pool (same pages, different queries and index lists)."""
    sets = [synth.batch_decode(seed=seed + k) for k in range(N_SETS)]
    # one pool for all sets: pool_seed and geometry come from the first set
    base = sets[0]
    for s in sets:
        s.pool_seed = base.pool_seed
    return sets


def new_token_batch(w: synth.DecodeWorkload, step_seed: int):
    rng = np.random.default_rng(10_000 + step_seed)
    lat = synth.bf16_from_f32(rng.standard_normal((w.n_rows, 512), dtype=np.float32))
    rope = synth.bf16_from_f32(rng.standard_normal((w.n_rows, 64), dtype=np.float32))
    slots = torch.from_numpy(rng.choice(w.num_slots, size=w.n_rows, replace=False).astype(np.int64))
    return lat, rope, slots


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------

def run_gpu(args):
    import nvfp4_kv_cache_sparse_gb300 as lib
    from synth.pool import fill_pool

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    lib.load()

    sets = make_sets(seed=rank * 100)
    w0 = sets[0]
    cache = fill_pool(lib.quantize_append, w0.num_slots, w0.record_bytes, w0.pool_seed, dev)
    qs = [s.q.to(dev) for s in sets]
    idxs = [s.indices.to(dev) for s in sets]
    news = [tuple(t.to(dev) for t in new_token_batch(w0, k)) for k in range(N_SETS)]
    splits = 0
    ws_bytes = lib.workspace_size(w0.B, w0.s_q, w0.h_q, w0.topk, w0.record_bytes, splits)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((w0.B, w0.s_q, w0.h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w0.B, w0.s_q, w0.h_q), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def append(k, s):
        lat, rope, slots = news[k % N_SETS]
        lib.quantize_append(lat, rope, slots, cache, dev_status=status, stream=s)

    def decode(k, s):
        lib.sparse_mla_decode(qs[k % N_SETS], cache, idxs[k % N_SETS], w0.sm_scale, out=out, lse=lse,
                              num_splits=splits, workspace=workspace, dev_status=status, stream=s)

    for k in range(args.warmup):
        append(k, stream)
        decode(k, stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    # The same library calls captured once into CUDA graphs: one graph holds a lap of all
    # N_SETS steps, so replaying it enqueues N_SETS steps in a few microseconds of host time and
    # every kernel is a programmatic dependent of the one before it (each starts its prologue
    # while its predecessor finishes); one graph per set holds a single step (for step counts
    # that are not whole laps), and one graph the lap's decode calls alone (for timing them).
    graphs = []
    cap = torch.cuda.Stream()
    g_lap = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_lap, stream=cap):
        for k in range(N_SETS):
            append(k, cap)
            decode(k, cap)
    g_decode_lap = torch.cuda.CUDAGraph()   # the decode calls of a lap alone, back to back
    with torch.cuda.graph(g_decode_lap, stream=cap):
        for k in range(N_SETS):
            decode(k, cap)
    for k in range(N_SETS):
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=cap):
            append(k, cap)
            decode(k, cap)
        graphs.append(g_step)

    def run_steps(k0, n):
        """Steps k0 .. k0 + n - 1: single-step graphs up to a lap boundary, then whole laps."""
        k = k0
        while k < k0 + n and k % N_SETS != 0:
            graphs[k % N_SETS].replay()
            k += 1
        while k + N_SETS <= k0 + n:
            g_lap.replay()
            k += N_SETS
        while k < k0 + n:
            graphs[k % N_SETS].replay()
            k += 1

    run_steps(0, args.warmup)
    for k in range(args.warmup):
        g_decode_lap.replay()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    # ---- device-timed steps (inputs resident in HBM)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        start.record(stream)
        run_steps(args.warmup, args.steps)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        # the decode call alone: DECODE_CALLS_TIMED calls in laps of N_SETS back-to-back calls,
        # each lap between its own pair of events, whatever --steps is
        n_laps = DECODE_CALLS_TIMED // N_SETS
        lap_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_laps)]
        for a, b in lap_evs:
            a.record(stream)
            g_decode_lap.replay()
            b.record(stream)
        torch.cuda.synchronize()
    t_local = start.elapsed_time(end) / 1e3
    t_job = max_over_ranks(t_local, world, dev)
    decode_us_laps = sorted(a.elapsed_time(b) / N_SETS * 1e3 for a, b in lap_evs)
    decode_s = statistics.median(decode_us_laps) / 1e6
    pct = lambda f: float(np.percentile(decode_us_laps, f))   # noqa: E731
    clocks = sampler.summary()
    # kernels per call, as the library plans them for this shape on this device
    _, decode_launches = lib.decode_plan(w0.B, w0.s_q, w0.h_q, w0.topk, w0.record_bytes, splits)
    append_launches = 1

    # ---- end to end through the public API with host buffers: every step copies its inputs in
    # from pinned host memory and its result out. Device inputs and outputs are double-buffered
    # over three streams (copy in, compute, copy out), so step k+1's upload and step k-1's
    # download overlap step k's kernels, as a caller pipelining these calls would.
    # Each set's inputs (q, indices, the new tokens) sit in one pinned buffer and go up in one copy;
    # out and lse come back in one copy. The tensors the calls take are views of those buffers.
    packed, views = pack_layout, pack_views
    in_parts = [(tuple(t.shape), t.dtype) for t in (sets[0].q, sets[0].indices) + tuple(new_token_batch(w0, 0))]
    in_offs, in_bytes = packed(in_parts)
    res_parts = [(tuple(out.shape), out.dtype), (tuple(lse.shape), lse.dtype)]
    res_offs, res_bytes = packed(res_parts)
    host_in = []
    for k in range(N_SETS):
        buf = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        for v, t in zip(views(buf, in_parts, in_offs), (sets[k].q, sets[k].indices) + tuple(new_token_batch(w0, k))):
            v.copy_(t)
        host_in.append(buf)
    host_res = [torch.empty(res_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_res = [torch.empty(res_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_q, d_idx, d_lat, d_rope, d_slots = zip(*[views(d_in[b], in_parts, in_offs) for b in range(2)])
    d_out, d_lse = zip(*[views(d_res[b], res_parts, res_offs) for b in range(2)])
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    s_default = torch.cuda.current_stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer b uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]   # kernels done with buffer b
    ev_out = [torch.cuda.Event() for _ in range(2)]    # result of buffer b downloaded
    for e in ev_used + ev_out:
        e.record(stream)

    def e2e_step(k):
        j, b = k % N_SETS, k % 2
        torch.cuda.set_stream(s_in)
        s_in.wait_event(ev_used[b])
        d_in[b].copy_(host_in[j], non_blocking=True)
        ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        s_comp.wait_event(ev_out[b])
        lib.quantize_append(d_lat[b], d_rope[b], d_slots[b], cache, stream=s_comp)
        lib.sparse_mla_decode(d_q[b], cache, d_idx[b], w0.sm_scale, out=d_out[b], lse=d_lse[b],
                              num_splits=splits, workspace=workspace, stream=s_comp)
        ev_used[b].record(s_comp)
        torch.cuda.set_stream(s_out)
        s_out.wait_event(ev_used[b])
        host_res[b].copy_(d_res[b], non_blocking=True)
        ev_out[b].record(s_out)
        torch.cuda.set_stream(s_default)

    for k in range(args.warmup):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(s_in)
    for k in range(args.steps):
        e2e_step(k)
    for s_ in (s_comp, s_out):
        s_in.wait_stream(s_)
    e2.record(s_in)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(s2.elapsed_time(e2) / 1e3, world, dev)
    h2d, d2h = in_bytes, res_bytes   # bytes copied each step (the parts plus their alignment padding)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after timing")

    result = None
    if rank == 0:
        peaks, peak_src = load_peaks()
        flops, alg_bytes = roofline_numbers(w0)
        achieved = flops / decode_s / 1e12
        peak = float(peaks["bf16_tflops"])
        traffic = NCU_TRAFFIC.get(decode_source_hash())
        cpu = cpu_baseline(args, w0) if (world == 1 and not args.no_cpu_baseline) else None
        configs = None
        if world == 1 and not args.no_configs:
            configs = measure_configs(dev, args.config_iters)
        launches = decode_launches + append_launches
        result = {
            "metric": METRIC,
            "value": job_throughput(w0.n_rows * args.steps, world, t_job),
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": t_job / args.steps * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {
                "workload": w0.name,
                "batch": w0.B, "s_q": w0.s_q, "h_q": w0.h_q, "topk": w0.topk, "record_bytes": w0.record_bytes,
                "pool_slots": w0.num_slots, "page_tokens": synth.PAGE, "seq_len": int(w0.seq_lens[0]),
                "appended_tokens_per_step": w0.n_rows, "num_splits": "auto",
                "l2": f"inputs larger than L2: {N_SETS} rotating index/query sets gather "
                      f"{N_SETS * w0.n_rows * w0.topk * w0.record_bytes / 1e6:.0f} MB of records per lap",
                "parallelism": f"replicas x{world}",
                "launch": "device-timed steps replay CUDA graphs of the API calls (a lap of all input sets per graph); "
                          "e2e calls the API directly",
            },
            "roofline": {
                "bound": "tensor",
                "achieved": achieved,
                "peak": peak,
                "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": traffic,
                "kernel": "decode call (decode_pair_kernel, the splits merged inside it), CUDA events on the launch "
                          f"stream around {n_laps} laps of {N_SETS} back-to-back calls over the rotating inputs "
                          "(graph-replayed); median lap",
                "peak_source": f"{peak_src} bf16 burst",
                "decode_us": decode_s * 1e6,
                "decode_us_p10": pct(10),
                "decode_us_p90": pct(90),
                "decode_calls_timed": n_laps * N_SETS,
                "decode_kernels_per_call": decode_launches,
                "roofline_us": max(flops / (peak * 1e12), alg_bytes / (float(peaks["hbm_gbs"]) * 1e9)) * 1e6,
                "algorithmic_flops": flops,
                "algorithmic_bytes": alg_bytes,
            },
            "cpu_baseline": cpu,
            "e2e": {"value": job_throughput(w0.n_rows * args.steps, world, t_e2e), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
            "configs": configs,
        }
    barrier(world)
    return result


# ---------------------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------------------

class OracleStep:
    """The oracle's pass over sampled rows of one batch: append of their new tokens + decode
    (threads: OpenMP threads of the decode, 0 = all host cores)."""

    def __init__(self, w: synth.DecodeWorkload, rows: np.ndarray, threads: int = 0):
        import oracle
        self.oracle = oracle
        slots, q, idx = synth.compact_for_rows(w, rows)
        lat, rope = synth.pool_rows(w.pool_seed, torch.from_numpy(slots))
        self.cache = np.zeros((slots.size + rows.size, w.record_bytes), dtype=np.uint8)
        oracle.quantize_append(synth.bf16_bits(lat), synth.bf16_bits(rope), np.arange(slots.size), self.cache)
        self.q = synth.bf16_bits(q)
        self.idx = idx
        self.w = w
        nl, nr, _ = new_token_batch(w, 0)
        self.new_lat = synth.bf16_bits(nl)[: rows.size]
        self.new_rope = synth.bf16_bits(nr)[: rows.size]
        self.new_slots = np.arange(slots.size, slots.size + rows.size, dtype=np.int64)
        self.rows = rows.size
        self.threads = threads

    def __call__(self):
        self.oracle.quantize_append(self.new_lat, self.new_rope, self.new_slots, self.cache)
        self.oracle.sparse_mla_decode(self.q, self.cache, self.idx, self.w.sm_scale, threads=self.threads)
        return self.rows


def oracle_decode_rate(w: synth.DecodeWorkload, n_rows: int = 4, block_scales: bool = False) -> dict:
    """The oracle's decode rate on a sample of a configuration's query rows (CPU, fp64), for the
    sweep lines: records of the sampled rows' slots are built first and not timed."""
    import oracle
    rows = synth.sample_rows(w, min(n_rows, w.n_rows))
    slots, q, idx = synth.compact_for_rows(w, rows)
    lat, rope = synth.pool_rows(w.pool_seed, torch.from_numpy(slots))
    recs = oracle.quantize_records(synth.bf16_bits(lat), synth.bf16_bits(rope), w.record_bytes,
                                   block_scales=block_scales)
    sink = None if w.attn_sink is None else w.attn_sink.numpy()
    t0 = time.perf_counter()
    oracle.sparse_mla_decode(synth.bf16_bits(q), recs, idx, w.sm_scale, attn_sink=sink, block_scales=block_scales)
    el = time.perf_counter() - t0
    return {"oracle_query_tokens_per_s": rows.size / el, "oracle_cores": oracle.threads_available(),
            "oracle_sample": f"{rows.size} of {w.n_rows} query rows (all heads, all keys)"}


def oracle_append_rate(ww, n_tokens: int = 2048) -> dict:
    """The oracle's append rate on the first n_tokens of a write workload (CPU)."""
    import oracle
    n = min(n_tokens, ww.T)
    cache = np.zeros((n, ww.record_bytes), dtype=np.uint8)
    lat, rope = synth.bf16_bits(ww.latent[:n]), synth.bf16_bits(ww.rope[:n])
    t0 = time.perf_counter()
    oracle.quantize_append(lat, rope, np.arange(n, dtype=np.int64), cache)
    el = time.perf_counter() - t0
    return {"oracle_tokens_per_s": n / el, "oracle_sample": f"{n} of {ww.T} tokens"}


def cpu_baseline(args, w):
    import oracle
    rows = np.arange(w.n_rows)
    job = OracleStep(w, rows)
    t0 = time.perf_counter()
    done, reps = 0, 0
    while True:
        done += job()
        reps += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds or reps >= 50:
            break
    # the same oracle on one core: a bounded sample of rows (the whole step would take minutes)
    one = OracleStep(w, rows[: args.cpu_rows_1core], threads=1)
    t1 = time.perf_counter()
    done1, reps1 = 0, 0
    while True:
        done1 += one()
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= args.cpu_seconds / 2 or reps1 >= 50:
            break
    return {"value": done / el, "unit": UNIT, "cores": oracle.threads_available(), "kind": "oracle",
            "sample": f"{reps} x one full step ({w.n_rows} rows x {w.h_q} heads x {w.topk} keys, plus the "
                      f"{w.n_rows} appended tokens), fp64 C oracle, OpenMP over heads",
            "seconds": el,
            "single_core": {"value": done1 / el1, "unit": UNIT, "cores": 1,
                            "sample": f"{reps1} x {one.rows} of the step's rows (all heads, all keys) plus their "
                                      f"appended tokens, one OpenMP thread", "seconds": el1}}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    sets = make_sets(seed=0)
    w0 = sets[0]
    per_step = args.ref_rows
    jobs = [OracleStep(s, np.arange(k * per_step, (k + 1) * per_step) % s.n_rows) for k, s in enumerate(sets)]
    for k in range(args.warmup):
        jobs[k % N_SETS]()
    t0 = time.perf_counter()
    done = 0
    for k in range(args.steps):
        done += jobs[k % N_SETS]()
    el = time.perf_counter() - t0
    value = done / el
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w0.name, "batch": w0.B, "s_q": w0.s_q, "h_q": w0.h_q, "topk": w0.topk,
                   "record_bytes": w0.record_bytes, "pool_slots": w0.num_slots,
                   "rows_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads_available(), "kind": "oracle",
                         "sample": f"{per_step} of {w0.n_rows} query rows per step (all heads, all keys) "
                                   f"plus their appended tokens"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------------
# --sweep: every configuration of the pages' workloads, one JSON line each (not the bench line)
# ---------------------------------------------------------------------------------------

def _time_calls(fn, iters: int, flush=None) -> float:
    """Seconds per call. Warm (flush None): `iters` back-to-back calls between two CUDA events,
    the host running ahead of the device. Cold: `flush` (writes a buffer larger than L2) runs
    before every call outside its own event pair; the median call is returned."""
    if flush is None:
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.record()
        for _ in range(iters):
            fn()
        en.record()
        en.synchronize()
        return st.elapsed_time(en) * 1e-3 / iters
    times = []
    for _ in range(iters):
        flush()
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.record()
        fn()
        en.record()
        en.synchronize()
        times.append(st.elapsed_time(en) * 1e-3)
    return float(np.median(times))


DECODE_CONFIGS = (
    ("tiny_b1_h64_topk64_R352", lambda: synth.tiny_decode(seed=0)),
    ("varlen_b128_sq2_h64_topk2048_R352_sink", lambda: synth.varlen_decode(seed=0)),
    ("longctx_b64_sq1_h128_topk2048_R432", lambda: synth.long_context(seed=0)),
    ("prefill_b2_sq256_h128_topk2048_prefix16384_R352", lambda: synth.sparse_prefill(seed=0)),
    # the batch decode over 656-byte fp8 records (the NVFP4-vs-fp8 comparison)
    ("decode_b32_sq1_h128_topk2048_R656", lambda: dataclasses.replace(synth.batch_decode(seed=0), record_bytes=656)),
)


def measure_decode(w, dev, iters, flush, peaks):
    import nvfp4_kv_cache_sparse_gb300 as lib
    from synth.pool import fill_pool
    tflops, hbm = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
    cache = fill_pool(lib.quantize_append, w.num_slots, w.record_bytes, w.pool_seed, dev)
    q, idx = w.q.to(dev), w.indices.to(dev)
    sink = None if w.attn_sink is None else w.attn_sink.to(dev)
    out = torch.empty((w.B, w.s_q, w.h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.s_q, w.h_q), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lib.workspace_size(w.B, w.s_q, w.h_q, w.topk, w.record_bytes, 0)), dtype=torch.uint8,
                     device=dev)

    def call():
        lib.sparse_mla_decode(q, cache, idx, w.sm_scale, attn_sink=sink, out=out, lse=lse, workspace=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    with sampler:
        warm = _time_calls(call, iters)
        cold = _time_calls(call, iters, flush)
    flops, bytes_ = roofline_numbers(w)
    t_roof = max(bytes_ / (hbm * 1e9), flops / (tflops * 1e12))
    vflops, vbytes = roofline_numbers_valid_only(w)
    t_roof_valid = max(vbytes / (hbm * 1e9), vflops / (tflops * 1e12))
    res = {"kind": "decode", "query_tokens": w.n_rows, "us_per_call_warm": warm * 1e6, "us_per_call_cold": cold * 1e6,
           "query_tokens_per_s_cold": w.n_rows / cold, "roofline_us": t_roof * 1e6, "roofline_frac_cold": t_roof / cold,
           "roofline_frac_warm": t_roof / warm,
           "bound": "tensor" if flops / (tflops * 1e12) > bytes_ / (hbm * 1e9) else "hbm",
           "algorithmic_flops": flops, "algorithmic_bytes": bytes_,
           "valid_index_fraction": int((w.indices >= 0).sum()) / w.indices.numel(), "calls_timed": iters,
           "roofline_us_valid_only": t_roof_valid * 1e6, "roofline_frac_cold_valid_only": t_roof_valid / cold,
           "clocks": sampler.summary()}
    del cache
    torch.cuda.empty_cache()
    return res


def measure_write(ww, dev, iters, flush, peaks, producer=None, flush_clean=None):
    """The append (or, with a producer workload, the fused norm + rotary + append and the unfused
    path it replaces: torch norm and rotation into a bf16 intermediate, then the append)."""
    import nvfp4_kv_cache_sparse_gb300 as lib
    hbm = float(peaks["hbm_gbs"])
    cache = torch.full((ww.num_slots, ww.record_bytes), ww.fill_byte, dtype=torch.uint8, device=dev)
    lat, rope, slots = ww.latent.to(dev), ww.rope.to(dev), ww.slot_mapping.to(dev)
    if producer is None:
        def call():
            lib.quantize_append(lat, rope, slots, cache)
        bytes_ = ww.T * (512 * 2 + 64 * 2 + 8 + ww.record_bytes)
    else:
        pw = producer
        nw, pos = pw.norm_weight.to(dev), pw.positions.to(dev)
        cos, sin = pw.cos_table.to(dev), pw.sin_table.to(dev)

        def call():
            lib.norm_rope_quantize_append(lat, nw, pw.eps, rope, pos, cos, sin, pw.rotate_half, slots, cache)

        def unfused():
            y = torch.nn.functional.rms_norm(lat.float(), (512,), weight=nw.float(), eps=pw.eps).to(torch.bfloat16)
            c, s_ = cos[pos], sin[pos]
            a, b = rope[:, :32].float(), rope[:, 32:].float()
            r = torch.cat([a * c - b * s_, b * c + a * s_], dim=1).to(torch.bfloat16)
            lib.quantize_append(y, r, slots, cache)
        # + the position (8 B) and the token's cos / sin rows (256 B, from L2 for hot positions)
        bytes_ = ww.T * (512 * 2 + 64 * 2 + 8 + 8 + ww.record_bytes)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    with sampler:
        warm = _time_calls(call, iters)
        cold = _time_calls(call, iters, flush)
        unf = _time_calls(unfused, max(5, iters // 4), flush) if producer is not None else None
        clean = _time_calls(call, iters, flush_clean) if flush_clean is not None else None
    t_roof = bytes_ / (hbm * 1e9)
    res = {"kind": "quantize_append" if producer is None else "norm_rope_quantize_append", "tokens": ww.T,
           "us_per_call_warm": warm * 1e6, "us_per_call_cold": cold * 1e6, "tokens_per_s_cold": ww.T / cold,
           "achieved_gbs_cold": bytes_ / cold / 1e9, "roofline_us": t_roof * 1e6, "roofline_frac_cold": t_roof / cold,
           "bound": "hbm", "algorithmic_bytes": bytes_, "calls_timed": iters, "clocks": sampler.summary()}
    if clean is not None:
        # cold with a clean L2: the flush reads a 512 MB buffer instead of writing it, so no dirty
        # lines of the flush are written back to HBM while the call runs
        res["us_per_call_cold_clean_l2"] = clean * 1e6
        res["roofline_frac_cold_clean_l2"] = t_roof / clean
    if unf is not None:
        res["unfused_us_per_call_cold"] = unf * 1e6
        res["unfused_path"] = "torch rms_norm and rotation into a bf16 intermediate, then quantize_append"
    del cache
    torch.cuda.empty_cache()
    return res


def measure_configs(dev, iters) -> dict:
    """Every configuration besides the headline one, at N=1: cold and warm microseconds per call,
    roofline fraction and the clocks seen while timing it (the default line carries them)."""
    peaks, _ = load_peaks()
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    scrub_i = scrub.view(torch.int32)

    def flush():
        scrub.fill_(1)

    def flush_clean():
        scrub_i.sum()

    res = {}
    for name, make in DECODE_CONFIGS:
        res[name] = measure_decode(make(), dev, iters, flush, peaks)
    for R in (352, 656):
        ww = synth.write_path(seed=0, record_bytes=R)
        res[ww.name] = measure_write(ww, dev, iters, flush, peaks, flush_clean=flush_clean)
    pw = synth.producer_inputs(seed=0, record_bytes=352)
    res["norm_rope_" + pw.write.name] = measure_write(pw.write, dev, iters, flush, peaks, producer=pw,
                                                      flush_clean=flush_clean)
    del scrub
    torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """Every configuration, one JSON line each (not the bench line), with the oracle's rate on a
    sample of each."""
    dev = torch.device("cuda", 0)
    peaks, peak_src = load_peaks()
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # > L2: written before cold calls

    def flush():
        scrub.fill_(1)

    iters = max(5, args.sweep_iters)
    cfgs = (("decode_b32_sq1_h128_topk2048_R352", lambda: synth.batch_decode(seed=0)),) + DECODE_CONFIGS
    want = lambda name: args.sweep_filter is None or args.sweep_filter in name   # noqa: E731
    for name, make in cfgs:
        if not want(name):
            continue
        w = make()
        line = {"sweep": True, "workload": name, **measure_decode(w, dev, iters, flush, peaks), "peaks": peak_src,
                **oracle_decode_rate(w)}
        print(json.dumps(line), flush=True)
    # scale-layout comparison (FlashMLA PR 18, format block: the permuted scale placement is
    # credited with 10-12% of decode latency): the batch decode workload on two pools of the same
    # contents, one with permuted scales and one with block-order scales, timed in alternating
    # rounds in one process
    if want("scale_layout_decode_b32_sq1_h128_topk2048_R352"):
        run_scale_layout(args, dev, iters, flush)
    # write path (quantize-append of 65,536 tokens into a 262,144-slot pool), 352-byte records and
    # the 656-byte fp8 records they are compared with; then the fused producer
    for R in (352, 656):
        ww = synth.write_path(seed=0, record_bytes=R)
        if want(ww.name):
            print(json.dumps({"sweep": True, "workload": ww.name, **measure_write(ww, dev, iters, flush, peaks),
                              "peaks": peak_src, **oracle_append_rate(ww)}), flush=True)
    pw = synth.producer_inputs(seed=0, record_bytes=352)
    if want("norm_rope_" + pw.write.name):
        print(json.dumps({"sweep": True, "workload": "norm_rope_" + pw.write.name,
                          **measure_write(pw.write, dev, iters, flush, peaks, producer=pw), "peaks": peak_src}),
              flush=True)


def run_scale_layout(args, dev, iters, flush):
    import nvfp4_kv_cache_sparse_gb300 as lib
    from synth.pool import fill_pool
    w = synth.batch_decode(seed=0)
    q, idx = w.q.to(dev), w.indices.to(dev)
    out = torch.empty((w.B, w.s_q, w.h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.s_q, w.h_q), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lib.workspace_size(w.B, w.s_q, w.h_q, w.topk, w.record_bytes, 0)), dtype=torch.uint8,
                     device=dev)
    pools = {False: fill_pool(lib.quantize_append, w.num_slots, 352, w.pool_seed, dev),
             True: fill_pool(functools.partial(lib.quantize_append, block_scales=True), w.num_slots, 352,
                             w.pool_seed, dev)}
    times = {(blk, kind): [] for blk in pools for kind in ("warm", "cold")}
    for rnd in range(6):
        for blk in ((False, True) if rnd % 2 == 0 else (True, False)):
            def call(c=pools[blk], b=blk):
                lib.sparse_mla_decode(q, c, idx, w.sm_scale, out=out, lse=lse, workspace=ws, block_scales=b)

            for _ in range(3):
                call()
            torch.cuda.synchronize()
            times[(blk, "warm")].append(_time_calls(call, iters))
            times[(blk, "cold")].append(_time_calls(call, iters, flush))
    med = {k: float(np.median(v)) * 1e6 for k, v in times.items()}
    print(json.dumps({"sweep": True, "workload": "scale_layout_decode_b32_sq1_h128_topk2048_R352",
                      "kind": "decode_scale_layout",
                      "us_per_call_warm": {"permuted": med[(False, "warm")], "block_order": med[(True, "warm")]},
                      "us_per_call_cold": {"permuted": med[(False, "cold")], "block_order": med[(True, "cold")]},
                      "block_order_over_permuted_cold": med[(True, "cold")] / med[(False, "cold")],
                      "block_order_over_permuted_warm": med[(True, "warm")] / med[(False, "warm")],
                      "rounds": 6, "calls_per_round": iters}), flush=True)
    del pools
    torch.cuda.empty_cache()


def run_profile_config(name: str):
    """Four calls (three warm-up, then the one an ncu capture with `-s 3 -c 1` takes) of one
    configuration's kernel, untimed: the command the summaries under profiles/ were taken with."""
    import nvfp4_kv_cache_sparse_gb300 as lib
    from synth.pool import fill_pool
    lib.load()
    dev = torch.device("cuda", 0)
    if name in ("decode", "longctx", "varlen", "tiny", "prefill", "fp8"):
        make = {"decode": synth.batch_decode, "longctx": synth.long_context, "varlen": synth.varlen_decode,
                "tiny": synth.tiny_decode, "prefill": synth.sparse_prefill, "fp8": synth.batch_decode}[name]
        # varlen at B = 32 (a 0.78 GB pool) instead of 128 (3 GB), to keep the profiler's replays small
        w = make(seed=0, B=32) if name == "varlen" else make(seed=0)
        if name == "fp8":
            w = dataclasses.replace(w, record_bytes=656)
        cache = fill_pool(lib.quantize_append, w.num_slots, w.record_bytes, w.pool_seed, dev)
        q, idx = w.q.to(dev), w.indices.to(dev)
        sink = None if w.attn_sink is None else w.attn_sink.to(dev)

        def call():
            lib.sparse_mla_decode(q, cache, idx, w.sm_scale, attn_sink=sink)
    else:
        pw = synth.producer_inputs(seed=0, record_bytes=352)
        ww = pw.write if name == "producer" else synth.write_path(seed=0, record_bytes=352)
        cache = torch.full((ww.num_slots, 352), ww.fill_byte, dtype=torch.uint8, device=dev)
        lat, rope, slots = ww.latent.to(dev), ww.rope.to(dev), ww.slot_mapping.to(dev)
        nw, pos = pw.norm_weight.to(dev), pw.positions.to(dev)
        cos, sin = pw.cos_table.to(dev), pw.sin_table.to(dev)

        def call():
            if name == "append":
                lib.quantize_append(lat, rope, slots, cache)
            else:
                lib.norm_rope_quantize_append(lat, nw, pw.eps, rope, pos, cos, sin, pw.rotate_half, slots, cache)
    torch.cuda.synchronize()
    for _ in range(4):
        call()
    torch.cuda.synchronize()
    print(json.dumps({"profile_config": name, "calls": 4}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows-1core", type=int, default=2,
                    help="query rows of the single-core oracle sample in cpu_baseline")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave out the per-configuration measurements of the N=1 line")
    ap.add_argument("--config-iters", type=int, default=20)
    ap.add_argument("--sweep", action="store_true",
                    help="time every workload configuration (decode and write path), one JSON line each")
    ap.add_argument("--sweep-iters", type=int, default=20)
    ap.add_argument("--sweep-filter", default=None,
                    help="with --sweep: time only the configurations whose name contains this string")
    ap.add_argument("--profile-config", choices=["decode", "longctx", "varlen", "tiny", "prefill", "fp8", "append", "producer"],
                    default=None,
                    help="make four untimed calls of one configuration (for ncu captures) and exit")
    args = ap.parse_args()
    if args.profile_config:
        run_profile_config(args.profile_config)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)
    world, _, _ = dist_env()
    if world > 1 and args.impl == "gpu":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
