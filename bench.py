"""Benchmark: paged decode attention, SenseNova-style decode step on one GB300.

A step is one replay of the captured decode graph: 42 layers, each one fused
append + attention launch (32 q / 8 kv heads, head_dim 128, bf16, one
sequence behind an identity block table) at a given KV length.  The headline
is KV length 8192 in the 8192 bucket; a sweep over other lengths (each in its
own bucket's graph) is reported beside it.  L2 is flushed (256 MiB write)
before every timed step, outside the timed events.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS, HQ, HKV, D = 42, 32, 8, 128
HEADLINE_LEN = 8192
SWEEP = (256, 512, 1024, 2048, 4096, 6144, 8192)
METRIC = "paged decode attention µs/step and achieved HBM GB/s (% of peak) vs KV length"
WORKLOAD = ("SenseNova-style decode: 42 layers, 32 q / 8 kv heads, head_dim 128, bf16, one sequence, "
            "identity block table, KV length 8192 in the 8192 bucket, one captured graph per bucket")
KERNEL_SOURCES = ("paged_kv_decode_13_gb300/csrc/decode.cuh", "paged_kv_decode_13_gb300/csrc/attend.cuh",
                  "paged_kv_decode_13_gb300/csrc/common.cuh",
                  "paged_kv_decode_13_gb300/csrc/attend_inst.cu")
PROFILE = os.path.join(ROOT, "profiles", "decode_sensenova_8192_traffic.json")


def algorithmic_bytes_per_layer(L: int) -> int:
    """Bytes one layer's append + attention must move at KV length L.

    K and V of every live key (L * kv_heads * head_dim * 2 tensors * 2 B),
    the query (Hq * D * 2 B), the appended K/V row written once
    (2 * Hkv * D * 2 B), the fp32 output (Hq * D * 4 B), the block-table
    entries of the live pages (4 B each) and the segment entry (16 B)."""
    kv = L * HKV * D * 2 * 2
    q = HQ * D * 2
    app = 2 * HKV * D * 2
    out = HQ * D * 4
    table = 4 * ((L + 15) // 16)
    return kv + q + app + out + table + 16


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 10 ms, each sample stamped
    on arrival; the summary keeps the samples that arrived inside the marked
    timed region (or, when that region is shorter than the sampling
    interval, the one nearest to it)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 10):
        import threading
        self.proc, self.samples, self.t0, self.t1 = None, [], None, None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", str(interval_ms), "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        first = threading.Event()

        def read():
            for line in self.proc.stdout:
                self.samples.append((time.perf_counter(), line))
                first.set()

        self.reader = threading.Thread(target=read, daemon=True)
        self.reader.start()
        first.wait(timeout=5.0)  # sampling is running before the region starts

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_stop(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.reader.join(timeout=5)
        t0 = self.t0 if self.t0 is not None else -math.inf
        t1 = self.t1 if self.t1 is not None else math.inf
        inside = [line for t, line in self.samples if t0 <= t <= t1]
        where = "inside the timed region"
        if not inside and self.samples:  # region shorter than the interval: the nearest sample
            mid = (t0 + t1) / 2 if math.isfinite(t0) and math.isfinite(t1) else 0.0
            inside = [min(self.samples, key=lambda x: abs(x[0] - mid))[1]]
            where = "nearest to the timed region (shorter than the sampling interval)"
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in inside:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms), "samples_taken": where}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def bench_config(world: int) -> dict:
    """The workload both arms report on."""
    return {"workload": WORKLOAD, "kv_len": HEADLINE_LEN, "bucket": 8192, "layers": LAYERS, "q_heads": HQ,
            "kv_heads": HKV, "head_dim": D,
            "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
            "parallelism": f"replicas x{world} (one sequence per GPU)"}


# ---------------------------------------------------------------- GPU arm

def make_runner(pkv, L: int, seed: int, device, advance: bool = False, bucket: int = 0, flags: int = 0):
    import torch

    import workloads
    from paged_kv_decode_13_gb300.graph import DecodeGraphRunner, DecodeStep
    bucket = bucket or pkv.bucket_for(L)
    w = workloads.sensenova(L, bucket, num_layers=LAYERS, seed=seed, device=device)
    cache = pkv.PagedKVCache(w.k, w.v, w.block_table, bucket=bucket)
    step = DecodeStep(cache, HQ, advance=advance, flags=flags)
    for layer in range(LAYERS):
        step.q[layer].copy_(w.q[layer])
        step.k_new[layer].copy_(w.k_new[layer])
        step.v_new[layer].copy_(w.v_new[layer])
    step.seq_info.copy_(w.seq_info)
    runner = DecodeGraphRunner(step)
    runner.graph_for()
    torch.cuda.synchronize()
    return runner, w


def time_steps(runner, steps: int, warmup: int, flush, stream, sampler=None):
    import torch
    graph = runner.graph_for()
    for _ in range(warmup):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if sampler is not None:
        sampler.mark_start()
    for a, b in evs:
        flush()
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.mark_stop()
    return [a.elapsed_time(b) for a, b in evs]


def time_clone(pkv, device, flush, stream, reps: int = 10, warmup: int = 3):
    """pkv_seq_clone of an 8192-token prefix in all 42 layers (the admission of
    a request that shares it): ms per clone and the bytes it moves."""
    import torch
    pages = HEADLINE_LEN // 16
    k = [torch.zeros(2 * pages, 16, HKV, D, dtype=torch.bfloat16, device=device) for _ in range(LAYERS)]
    v = [torch.zeros(2 * pages, 16, HKV, D, dtype=torch.bfloat16, device=device) for _ in range(LAYERS)]
    for t in k + v:
        t.normal_()
    bt = torch.arange(2 * pages, dtype=torch.int32, device=device).view(2, pages)
    cache = pkv.PagedKVCache(k, v, bt, bucket=HEADLINE_LEN)
    err = pkv.new_err_flags(device)
    for _ in range(warmup):
        pkv.seq_clone(cache, 0, 1, HEADLINE_LEN, err, stream=stream)
    ts = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pkv.seq_clone(cache, 0, 1, HEADLINE_LEN, err, stream=stream)
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"seq_clone error flags {int(err.item()):#x}")
    ms = statistics.median([a.elapsed_time(b) for a, b in ts])
    moved = 2 * 2 * LAYERS * HEADLINE_LEN * HKV * D * 2  # K and V, read and written
    del k, v, cache
    return ms, moved


def workload_bytes_flops(w):
    """Algorithmic bytes and flops of one fused append + attention launch over
    workload w: K and V of every key some row of a segment reads (per kv
    head), q, the appended rows, the fp32 output, the touched table entries
    and the segment entries; flops 4 * D per (query head, row, visible key)."""
    eb = w.k[0].element_size()
    kv = q = app = out = table = flops = 0
    for q0, ql, col, kend in w.seq_info.tolist():
        first = kend - ql
        newest0 = first if w.causal else kend - 1
        lo = max(0, newest0 - w.window + 1) if w.window > 0 else 0
        kv += (kend - lo) * w.kv_heads * w.head_dim * 2 * eb
        table += 4 * ((kend + 15) // 16 - lo // 16)
        for i in range(ql):
            p = first + i
            hi = p + 1 if w.causal else kend
            rlo = max(0, (p if w.causal else kend - 1) - w.window + 1) if w.window > 0 else 0
            flops += 4 * w.q_heads * w.head_dim * (hi - rlo)
        q += ql * w.q_heads * w.head_dim * eb
        app += 2 * ql * w.kv_heads * w.head_dim * eb
        out += ql * w.q_heads * w.head_dim * 4
    return kv + q + app + out + table + 16 * w.num_segments, flops


CONFIGS = (
    ("batched", "batched varlen: S=32, lengths U[1,16384], shuffled shared-pool tables, GQA 32:8, D 128, bf16, "
     "q_len 1", "batched", dict(S=32, max_len=16384)),
    ("verify_causal", "spec verify, causal: S=16, q_len U[1,16] aligned to kv_end, GQA 64:8, D 128, bf16, "
     "KV U[256,8192]", "spec_verify", dict(S=16, max_q=16, len_lo=256, len_hi=8192, causal=True)),
    ("verify_noncausal", "spec verify, non-causal draft blocks: same shapes, causal off",
     "spec_verify", dict(S=16, max_q=16, len_lo=256, len_hi=8192, causal=False)),
    ("long_context", "long context, full causal: S=4, KV 131072 flat, GQA 32:4, D 256, bf16, q_len 1",
     "long_context", dict(S=4, kv_len=131072)),
    ("long_context_ring", "long context, window 4096 over a 4096-row ring: S=4, KV 131072, GQA 32:4, D 256, "
     "bf16, q_len 1", "long_context", dict(S=4, kv_len=131072, window=4096, ring_rows=4096)),
)


def time_configs(pkv, device, flush, stream, peak: float, seed: int, reps: int = 50, warmup: int = 5, only=None,
                 flags: int = 0):
    """The other workloads of the scope table, one fused append + attention
    call each (one launch), L2 flushed before every timed call: median µs,
    algorithmic GB/s and its fraction of the copy peak."""
    import torch

    import workloads
    res = []
    for key, name, gen, kw in CONFIGS:
        if only is not None and key != only:
            continue
        w = getattr(workloads, gen)(seed=seed, device=device, **kw)
        cache = pkv.PagedKVCache(w.k, w.v, w.block_table, ring_rows=w.ring_rows, bucket=w.bucket)
        q, kn, vn, si = w.q[0], w.k_new[0], w.v_new[0], w.seq_info
        out = torch.empty(w.total_rows, w.q_heads, w.head_dim, device=device)
        err = pkv.new_err_flags(device)
        max_kv = int(si[:, 3].max().item())

        def call():
            pkv.append_attend(cache, 0, q, kn, vn, si, out, err, w.max_q_len, max_kv, w.scale, w.causal,
                              w.window, stream=stream, flags=flags)

        for _ in range(warmup):
            flush()
            call()
        evs = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        if int(err.item()):
            raise RuntimeError(f"{name}: device error flags {int(err.item()):#x}")
        ms = statistics.median([a.elapsed_time(b) for a, b in evs])
        nbytes, flops = workload_bytes_flops(w)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res.append({"key": key, "workload": name, "us": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                    "frac_of_peak": round(gbs / peak, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 2)})
        del w, cache, q, kn, vn, si, out
        torch.cuda.empty_cache()
    return res


def time_e2e(pkv, steps: int, warmup: int, flush, stream, seed: int, device):
    """End to end through the public API with host buffers.  Per step: one
    pinned host -> device copy of the step's rows (every layer's q, k_new and
    v_new), one replay of the captured step, which appends, attends and then
    advances kv_end on the device (so the segment table is written by the
    host once, before the first step), and one device -> host copy of every
    layer's output, all inside the timed events.  The lengths start
    warmup + steps - 1 below the headline length, so the last timed step
    runs at it.  Returns the step times, the bytes copied each way per step
    and the first and last KV length timed."""
    import torch
    first = HEADLINE_LEN - (warmup + steps) + 1
    runner, w = make_runner(pkv, first, seed, device, advance=True, bucket=pkv.bucket_for(HEADLINE_LEN))
    del w
    st = runner.step_bufs
    host_in = st.step_inputs.cpu().pin_memory()
    host_out = torch.empty(st.outputs.shape, dtype=st.outputs.dtype).pin_memory()
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    graph = runner.graph_for()

    def one():
        st.step_inputs.copy_(host_in, non_blocking=True)
        graph.replay()
        host_out.copy_(st.outputs, non_blocking=True)

    for _ in range(warmup):
        flush()
        one()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        one()
        b.record(stream)
    torch.cuda.synchronize()
    if int(st.err.item()):
        raise RuntimeError(f"e2e: device error flags {int(st.err.item()):#x}")
    last = int(st.seq_info[0, 3].item()) - 1
    assert last == HEADLINE_LEN, last
    del runner
    return [a.elapsed_time(b) for a, b in evs], h2d, d2h, first + warmup, last


def oracle_layer_seconds(q, k, v, L: int, kv_heads: int = HKV) -> float:
    """Seconds the fp64 C oracle takes for the first `kv_heads` kv heads (and
    their query heads) of one layer at KV length L; input widening excluded."""
    import numpy as np

    from oracle import oracle as orc
    g = HQ // HKV
    nb = (L + 15) // 16
    qd = np.ascontiguousarray(q[:, :kv_heads * g].double().numpy())
    kd = np.ascontiguousarray(k[:nb, :, :kv_heads].double().numpy())
    vd = np.ascontiguousarray(v[:nb, :, :kv_heads].double().numpy())
    si = np.array([[0, 1, 0, L]], np.int32)
    bt = np.arange(nb, dtype=np.int32)[None]
    t0 = time.perf_counter()
    orc.attend(qd, kd, vd, bt, si, 1 / math.sqrt(D))
    return time.perf_counter() - t0


def cpu_baseline_sample(layers, L: int, seconds: float = 12.0):
    """Whole layers of the step through the oracle on this host (one thread),
    cycling over the given layers until `seconds` of oracle time; returns the
    time scaled to the full 42-layer step in µs, and the layers run."""
    spent, done = 0.0, 0
    while True:
        q, k, v = layers[done % len(layers)]
        spent += oracle_layer_seconds(q, k, v, L)
        done += 1
        if spent >= seconds or done >= 4 * LAYERS:
            break
    return spent / done * LAYERS * 1e6, done


def _oracle_worker(job):
    """One host core: whole layers of a single-sequence KV-8192 step through
    the oracle from wall time `start_at` for `seconds`; returns the layers
    finished inside that window."""
    seed, start_at, seconds = job
    import numpy as np
    import torch
    torch.set_num_threads(1)
    import workloads
    from oracle import oracle as orc
    w = workloads.sensenova(HEADLINE_LEN, HEADLINE_LEN, num_layers=1, seed=seed, device="cpu")
    nb = HEADLINE_LEN // 16
    qd = np.ascontiguousarray(w.q[0].double().numpy())
    kd = np.ascontiguousarray(w.k[0].double().numpy())
    vd = np.ascontiguousarray(w.v[0].double().numpy())
    si = np.array([[0, 1, 0, HEADLINE_LEN]], np.int32)
    bt = np.arange(nb, dtype=np.int32)[None]
    while time.time() < start_at:
        time.sleep(0.001)
    done = 0
    while True:
        orc.attend(qd, kd, vd, bt, si, 1 / math.sqrt(D))
        if time.time() > start_at + seconds:
            return done
        done += 1


def cpu_baseline_all_cores(seconds: float = 8.0):
    """The oracle on every host core at once (one process per core, started
    with spawn): µs per 42-layer step from the layers all cores finish in a
    common window, and the core count."""
    import multiprocessing as mp
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    start_at = time.time() + 20.0
    with mp.get_context("spawn").Pool(n) as pool:
        done = sum(pool.map(_oracle_worker, [(i, start_at, seconds) for i in range(n)]))
    return (seconds / (done / LAYERS) * 1e6 if done else None), n, done


def gpu_arm(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as pkv

    stream = torch.cuda.current_stream()
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def flush():
        scratch.fill_(1)

    peak, peak_kind = load_peaks()

    # Headline: KV length 8192.
    runner, w = make_runner(pkv, HEADLINE_LEN, seed=rank, device=device, flags=args.flags)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(device.index or 0)
    times = time_steps(runner, args.steps, args.warmup, flush, stream, sampler=sampler)
    clocks = sampler.stop()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = statistics.mean(times)
    qs = statistics.quantiles(times, n=10) if len(times) >= 2 else [times[0]] * 9
    pct = {"p10": round(qs[0] * 1e3, 2), "p50": round(statistics.median(times) * 1e3, 2), "p90": round(qs[8] * 1e3, 2)}
    ms = reduce_max(ms, world, device)
    err = int(runner.step_bufs.err.item())
    if err:
        raise RuntimeError(f"device error flags {err:#x}")
    launches_per_step = runner.step_bufs.launch_count()
    bytes_layer = algorithmic_bytes_per_layer(HEADLINE_LEN)
    per_launch_ms = ms / launches_per_step
    achieved = bytes_layer / (per_launch_ms * 1e-3) / 1e9
    step_gbs = bytes_layer * LAYERS / (ms * 1e-3) / 1e9

    e2e_steps = min(max(args.steps // 4, 10), 200)
    e2e_times, h2d, d2h, e2e_lo, e2e_hi = time_e2e(pkv, e2e_steps, args.warmup, flush, stream, rank, device)
    e2e_ms = reduce_max(statistics.mean(e2e_times), world, device)

    # CPU oracle baseline on a bounded sample of the same step's layers.
    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu:
        layers = [(w.q[i].cpu(), w.k[i].cpu(), w.v[i].cpu()) for i in range(min(LAYERS, 6))]
        cpu_us, done = cpu_baseline_sample(layers, HEADLINE_LEN, seconds=args.cpu_seconds)
        cpu = {"value": round(cpu_us, 1), "unit": "µs/step", "cores": 1, "kind": "oracle",
               "sample": f"{done} whole layers (cycling over 6 of the step's 42) at KV length {HEADLINE_LEN} "
                         f"through the fp64 C oracle on one thread, mean per layer scaled to 42 layers"}
        all_us, ncores, ndone = cpu_baseline_all_cores()
        if all_us:
            cpu_all = {"value": round(all_us, 1), "unit": "µs/step", "cores": ncores, "kind": "oracle",
                       "sample": f"{ndone} whole layers at KV length {HEADLINE_LEN} finished by {ncores} processes "
                                 f"(one per host core) in a common 8 s window, scaled to 42 layers"}
    del runner, w
    torch.cuda.empty_cache()

    by_len = {}
    if not args.no_sweep:
        for L in SWEEP:
            r, _ = make_runner(pkv, L, seed=rank, device=device, flags=args.flags)
            t = time_steps(r, max(args.steps // 4, 20), args.warmup, flush, stream)
            m = reduce_max(statistics.median(t), world, device)
            gbs = algorithmic_bytes_per_layer(L) * LAYERS / (m * 1e-3) / 1e9
            by_len[str(L)] = {"bucket": pkv.bucket_for(L), "us_per_step": round(m * 1e3, 2),
                              "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
            del r
            torch.cuda.empty_cache()

    clone = None
    if not args.no_sweep:
        cms, moved = time_clone(pkv, device, flush, stream)
        cms = reduce_max(cms, world, device)
        cgbs = moved / (cms * 1e-3) / 1e9
        clone = {"what": f"pkv_seq_clone of a {HEADLINE_LEN}-token prefix in all {LAYERS} layers (K and V read and "
                         f"written)", "ms": round(cms, 4), "bytes": moved, "gbs": round(cgbs, 1),
                 "frac_of_peak": round(cgbs / peak, 4)}
        torch.cuda.empty_cache()

    by_config = None
    if not args.no_sweep:
        by_config = time_configs(pkv, device, flush, stream, peak, seed=rank, flags=args.flags)

    traffic = None
    if os.path.exists(PROFILE):
        with open(PROFILE) as f:
            prof = json.load(f)
        if prof.get("kernel_hash") == kernel_hash():
            traffic = prof.get("dram_bytes_per_launch")

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(ms * 1e3, 2),
            "unit": "µs/step",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 5),
            "step_us_percentiles": pct,
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded torch normal draws; q ~ N(0,1), K/V ~ N(0,1)/sqrt(128))",
            "config": bench_config(world),
            "hbm_gbs": round(step_gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": f"{peak_kind} (STREAM-style copy)",
                         "kernel": "decode_kernel (fused append + split-K attention, 16-CTA clusters; 6 warps x 2 stages at this bucket), one launch per layer",
                         "algorithmic_bytes_per_launch": bytes_layer,
                         "launch_ms": round(per_launch_ms, 6)},
            "by_kv_len": by_len,
            "seq_clone": clone,
            "by_config": by_config,
            "e2e": {"value": round(e2e_ms * 1e3, 2), "unit": "µs/step", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "kv_len": f"{e2e_lo}..{e2e_hi}, advanced on the device by the captured step",
                    "copies": "per step one pinned H2D of every layer's q, k_new, v_new and one D2H of every "
                              "layer's output; the segment table is written once, before the first step"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
        }
        if args.flags:
            line["config"]["attention_flags"] = args.flags
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def config_only(key: str, flags: int = 0):
    """One workload of the scope table, 3 + 3 calls, one JSON line (no
    headline): the command the profiler summaries capture."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as pkv
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    peak, _ = load_peaks()
    res = time_configs(pkv, device, lambda: scratch.fill_(1), torch.cuda.current_stream(), peak, seed=0, reps=3,
                       warmup=3, only=key, flags=flags)
    res[0]["flags"] = flags
    print(json.dumps(res[0]), flush=True)


def decode_layer_only(L: int, flags: int = 0):
    """One layer of the headline step (fused append + attention of one token,
    GQA 32:8, D 128) at KV length L, 3 + 3 launches with L2 flushed before
    each, one JSON line: the command the decode profiler summaries capture."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as pkv

    import workloads
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    peak, _ = load_peaks()
    bucket = pkv.bucket_for(L)
    w = workloads.sensenova(L, bucket, num_layers=1, seed=0, device=device)
    cache = pkv.PagedKVCache(w.k, w.v, w.block_table, bucket=bucket)
    out = torch.empty(w.total_rows, w.q_heads, w.head_dim, device=device)
    err = pkv.new_err_flags(device)
    stream = torch.cuda.current_stream()
    evs = []
    for i in range(6):
        scratch.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pkv.append_attend(cache, 0, w.q[0], w.k_new[0], w.v_new[0], w.seq_info, out, err, 1, L, w.scale, w.causal,
                          w.window, stream=stream, flags=flags)
        b.record(stream)
        if i >= 3:
            evs.append((a, b))
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"device error flags {int(err.item()):#x}")
    ms = statistics.median([a.elapsed_time(b) for a, b in evs])
    gbs = algorithmic_bytes_per_layer(L) / (ms * 1e-3) / 1e9
    print(json.dumps({"decode_layer": L, "flags": flags, "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                      "frac_of_peak": round(gbs / peak, 4)}), flush=True)


# ---------------------------------------------------------------- reference arm (CPU oracle)

def reference_arm(args):
    """The oracle as it stands on whole steps of the headline workload: per
    step, for each of the 42 layers, the oracle's append of the step's row
    and its attention over all 8 kv heads at KV length 8192, on one host
    thread.  Nothing is sampled or scaled; if the requested steps would take
    more than a few minutes the step count is cut (never the work per step)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import torch

    import workloads
    from oracle import oracle as orc
    orc.build()
    torch.set_num_threads(max(1, min(8, os.cpu_count() or 1)))
    w = workloads.sensenova(HEADLINE_LEN, HEADLINE_LEN, num_layers=LAYERS, seed=0, device="cpu")
    si = w.seq_info.numpy()
    bt = w.block_table.numpy()
    scale = 1 / math.sqrt(D)
    layers = []
    for i in range(LAYERS):
        kb = w.k[i].view(torch.int16).numpy().copy()
        vb = w.v[i].view(torch.int16).numpy().copy()
        kn = w.k_new[i].view(torch.int16).numpy()
        vn = w.v_new[i].view(torch.int16).numpy()
        assert orc.append(kb, vb, bt, si, kn, vn) == 0   # the pools the attention reads hold the step's row
        layers.append((kb, vb, kn, vn, w.q[i].double().numpy(),
                       torch.from_numpy(kb).view(torch.bfloat16).double().numpy(),
                       torch.from_numpy(vb).view(torch.bfloat16).double().numpy()))
    del w

    def one_step() -> float:
        t = 0.0
        for kb, vb, kn, vn, q, kd, vd in layers:
            t0 = time.perf_counter()
            orc.append(kb, vb, bt, si, kn, vn)
            orc.attend(q, kd, vd, bt, si, scale)
            t += time.perf_counter() - t0
        return t

    budget_s = 240.0
    start = time.perf_counter()
    first = one_step()
    for _ in range(args.warmup - 1):
        one_step()
    left = budget_s - (time.perf_counter() - start)
    steps = max(1, min(args.steps, int(left / max(first, 1e-6))))
    per = [one_step() * 1e6 for _ in range(steps)]
    us = statistics.mean(per)
    sample = (f"whole steps: per step {LAYERS} layers x (the oracle's one-row append + its fp64 attention over all "
              f"{HKV} kv heads at KV length {HEADLINE_LEN}), one host thread, C oracle built -O2; "
              f"{steps} timed steps after {args.warmup} warm-up")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "µs/step", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded torch normal draws; "
        "q ~ N(0,1), K/V ~ N(0,1)/sqrt(128))",
        "config": bench_config(world),
        "cpu_baseline": {"value": round(us, 1), "unit": "µs/step", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "µs/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if steps != args.steps:
        line["steps_requested"] = args.steps
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--config-only", choices=[c[0] for c in CONFIGS],
                    help="time only this workload's call (3 warm-up + 3 timed calls; for profiler runs)")
    ap.add_argument("--decode-layer", type=int, default=0, metavar="L",
                    help="time only one headline layer at KV length L (3 warm-up + 3 timed launches; for profiler runs)")
    ap.add_argument("--flags", type=int, default=0,
                    help="attention flags of every timed call (1: CUDA-core kernels, 8: mma.sync tile for wide groups)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        reference_arm(args)
    elif args.config_only:
        config_only(args.config_only, args.flags)
    elif args.decode_layer:
        decode_layer_only(args.decode_layer, args.flags)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
