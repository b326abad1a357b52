"""Benchmark: the Llama-3-8B-shaped 1-bit (Q1_0) decode matmul set, batch 1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over the 225 products of a decode
token (32 layers x q, k, v, o, gate, up, down + lm_head), each with its own
activation vector: q8_0 quantization of the f32 activation and the Q1_0
matrix-vector product.  The timed schedule is one q1_0_gemv_multi launch per
step (quantization fused), captured as a CUDA graph and replayed; the same work
is also timed as the launches a decode step's data dependencies allow
("grouped", 129), one launch per product ("decode", 225) and separate
quantize + product launches ("separate", 450).  Weights (1.055 GB of Q1_0
blocks) are packed once and stay resident; every step streams all of them,
more than the 126 MB L2, so no step reuses another's cached bytes.

Printed (rank 0, one JSON line):
  value       whole-job weight GB/s = n_gpus * weight bytes / max-over-ranks step time
  us_per_set  microseconds per decode matmul set on one GPU
  roofline    the product kernel (one launch per step): algorithmic bytes per
              launch / launch time vs the measured HBM peak
  e2e         same metric with the activations read from pinned host memory
              and the outputs written back to it inside every timed step
  cpu_baseline  the threaded CPU oracle timed over the whole set once (rank 0, N = 1 only)
  parity      that oracle pass's outputs against every output of the timed step
Multi-GPU: independent replicas (the product shards by rows, but this workload
is one GPU's; N GPUs run N copies), scaling "weak".

--impl reference times the CPU oracle (the definition the CUDA path must match
bit for bit) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("Q1_0 GEMV weight GB/s and % of HBM peak; µs per 8B-shaped decode matmul set")
WORKLOAD = "llama3-8b-shaped Q1_0 decode matmul set, batch 1 (225 products)"


# ------------------------------------------------------------- helpers ----
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the streaming kernel's code with comments and blank space
    removed: a recorded ncu capture stays valid across comment edits and is
    dropped by any change to the code itself."""
    import re
    h = hashlib.sha256()
    for rel in ("decode_q1_gemv_gb300/csrc/multi.cu", "decode_q1_gemv_gb300/csrc/table.cuh",
                "decode_q1_gemv_gb300/csrc/common.cuh", "decode_q1_gemv_gb300/csrc/q2.cuh",
                "decode_q1_gemv_gb300/csrc/formats.cuh"):
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM bytes of the product kernel from the committed ncu summary,
    valid only while the kernel source is unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", "q1_0_gemv_decode_set_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch_avg")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for _, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- CPU baseline --
def cpu_oracle_set(ds, gpu_out, threads: int, passes: int = 4):
    """The CPU baseline and the parity check of the timed step: the threaded
    oracle (q8_0 quantization + product) over every product of the decode set
    `ds`, on the same seeded inputs, `passes` times (about 10 s of CPU work
    for the full set), timed; and every output of the first pass compared bit
    for bit with `gpu_out`, the device's output buffer after one replay of the
    timed step.  Returns (weight GB/s, description, threads, parity record)."""
    import numpy as np

    import oracle

    oracle.build()
    elapsed, first_pass, checked, mismatches, first = 0.0, 0.0, 0, 0, None
    for i, (name, rows, n) in enumerate(ds.shapes):
        blocks, x = ds.host_blocks(i), ds.host_x(i)
        for k in range(passes):
            t0 = time.perf_counter()
            q, d = oracle.q8_quantize(x[None, :])
            res = oracle.gemv_threaded(blocks, q[0], d[0], threads)
            dt = time.perf_counter() - t0
            elapsed += dt
            if k == 0:
                first_pass += dt
                want, done = res
        got = gpu_out[ds.out_off[i]:ds.out_off[i] + rows]
        bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
        checked += rows
        mismatches += int(bad.size) + (rows - int(done))
        if first is None and (bad.size or done != rows):
            first = f"{name} row {int(bad[0]) if bad.size else int(done)}"
        del blocks
    gbs = passes * ds.weight_bytes / elapsed / 1e9
    desc = (f"the whole decode set {passes} times ({len(ds.shapes)} products, {ds.weight_bytes / 1e6:.1f} MB of "
            f"weights each time): q8_0 quantization + threaded oracle product, {threads} threads, {elapsed:.1f} s")
    parity = {"checked": checked, "mismatches": mismatches, "oracle_s": round(first_pass, 2),
              "compared": "every output of the timed step (one more replay of its graph) against the threaded "
                          "oracle on the same seeded inputs, f32 bits equal"}
    if first:
        parity["first_mismatch"] = first
    return gbs, desc, threads, parity


def cpu_context(seed: int = 3):
    """Host-side context for the CPU baseline: the single-thread oracle on the
    256x1024 and 4096x4096 products, on 14336x4096 with 16 vectors and on layer
    0 of the decode set; and a streaming read of a 768 MiB buffer (far larger
    than the caches) at 1..all threads, the memory floor a CPU decode is held
    to (bankML "docs/modules/par.md", benchmarks: bench_memory_floor)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    from decode_q1_gemv_gb300 import synth

    oracle.build()
    single = {}

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return (time.perf_counter() - t0) * 1e6

    for name, rows, n, nvec, outl in (("gemv_256x1024", 256, 1024, 1, 0.0), ("gemv_4096x4096", 4096, 4096, 1, 0.01),
                                      ("b16_14336x4096", 14336, 4096, 16, 0.0)):
        blocks = synth.weight_blocks(synth.rng_for(seed, rows, n, 0), rows, n)
        x = synth.activations(synth.rng_for(seed, rows, n, 1), nvec, n, outliers=outl)
        q, d = oracle.q8_quantize(x)
        fn = (lambda: oracle.gemv(blocks, q[0], d[0])) if nvec == 1 else (lambda: oracle.gemm(blocks, q, d))
        single[name] = round(timed(fn), 1)
    layer = [(synth.weight_blocks(synth.rng_for(seed, i, 0), rows, n), synth.activations(synth.rng_for(seed, i, 1), 1, n))
             for i, (_, rows, n) in enumerate(synth.decode_set_shapes()[:7])]

    def one_layer():
        for blocks, x in layer:
            q, d = oracle.q8_quantize(x)
            oracle.gemv(blocks, q[0], d[0])
    single["decode_set_layer0"] = round(timed(one_layer), 1)

    buf = np.ones(768 * 1024 * 1024 // 8, dtype=np.float64)
    floor = {}
    ncpu = os.cpu_count() or 1
    for t in sorted({1, 2, 4, 8, ncpu} & set(range(1, ncpu + 1))):
        parts = np.array_split(buf, t)
        with cf.ThreadPoolExecutor(t) as ex:
            list(ex.map(np.sum, parts))  # warm
            t0 = time.perf_counter()
            list(ex.map(np.sum, parts))
            dt = time.perf_counter() - t0
        floor[str(t)] = round(buf.nbytes / dt / 1e9, 2)
    del buf
    return {"oracle_single_thread_us": single, "memory_floor_read_gbs_by_threads": floor,
            "memory_floor_buffer_bytes": 768 * 1024 * 1024}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from decode_q1_gemv_gb300 import synth

    oracle.build()
    threads = os.cpu_count() or 1
    shapes = synth.decode_set_shapes()[:7]  # layer 0: q, k, v, o, gate, up, down
    inputs = []
    for i, (name, rows, n) in enumerate(shapes):
        blocks = synth.weight_blocks(synth.rng_for(3, i, 0), rows, n)
        x = synth.activations(synth.rng_for(3, i, 1), 1, n)
        inputs.append((blocks, x))
    sample_bytes = sum(rows * n * 18 // 128 for _, rows, n in shapes)

    def one_step():
        for blocks, x in inputs:
            q, d = oracle.q8_quantize(x)
            oracle.gemv_threaded(blocks, q[0], d[0], threads)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = sample_bytes / dt / 1e9
    desc = (f"each step: layer 0 of the decode set (7 products, {sample_bytes / 1e6:.1f} MB of weights), "
            f"q8_0 quantization + threaded oracle product, {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "layer 0 (7 products)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- ours -----
def max_over_ranks(v: float, world: int, dist=None, device=None) -> float:
    """Maximum of a per-rank float over all ranks (the rank's own value at N=1)."""
    if world == 1:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _time_graph(graph, reps, stream):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# The other configurations (single products and the batched product), timed
# one launch at a time with L2 flushed before each: cold-L2 median of `reps`.
OTHER_CONFIGS = (
    # name, rows, n, vectors, scale distribution, outlier fraction
    ("gemv_256x1024", 256, 1024, 1, "halfnormal", 0.0),
    ("gemv_4096x4096", 4096, 4096, 1, "halfnormal", 0.01),
    ("b16_14336x4096", 14336, 4096, 16, "halfnormal", 0.0),
    ("b16_4096x14336", 4096, 14336, 16, "halfnormal", 0.0),
    ("b64_128256x4096", 128256, 4096, 64, "lognormal", 0.0),
    ("b64_4096x14336", 4096, 14336, 64, "lognormal", 0.0),
)


# Roof of the batched product: the definition's chain needs at least 5 f32
# operations per lane, block and vector (d1*s, three fma with d1, the outer fma
# with d0) when the integer lane sums come for free: 5/16 per weight and vector
# on the CUDA cores' f32 pipes (128 lanes per SM per clock).  The tensor-core
# kernel takes most of the chain into its MMAs, so it is measured against the
# same roof (it could exceed it).
CHAIN_OPS_PER_WEIGHT_VECTOR = 5.0 / 16.0


def fp32_roof_ops_per_s(sm_mhz=None):
    import torch
    props = torch.cuda.get_device_properties(0)
    mhz = sm_mhz or 2070.0
    return props.multi_processor_count * 128 * mhz * 1e6


def time_other_configs(dev, reps: int = 15, only=None):
    import torch
    from decode_q1_gemv_gb300 import binding, synth

    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2
    stream = torch.cuda.current_stream(dev)
    roof = fp32_roof_ops_per_s()
    res = {}
    for ci, (name, rows, n, nvec, scale, outl) in enumerate(OTHER_CONFIGS):
        if only and name not in only:
            continue
        blocks = synth.weight_blocks(synth.rng_for(11, ci, 0), rows, n, scale)
        x = synth.activations(synth.rng_for(11, ci, 1), nvec, n, outliers=outl)
        packed = binding.pack(torch.from_numpy(blocks).to(dev), rows, n)
        q, d = binding.quantize(torch.from_numpy(x).to(dev))
        out = torch.empty((nvec, rows), dtype=torch.float32, device=dev)

        def launch():
            if nvec == 1:
                binding.gemv(packed, rows, n, q[0], d[0], out[0])
            else:
                binding.gemm_small(packed, rows, n, q, d, out)

        def cold_median():
            for _ in range(3):
                launch()
            ts = []
            for _ in range(reps):
                flush.add_(1.0)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                launch()
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            ts.sort()
            return ts[len(ts) // 2], ts[0]

        us, us_min = cold_median()
        wbytes = rows * n * 18 // 128
        entry = {"rows": rows, "n": n, "vectors": nvec, "us": round(us, 2), "us_min": round(us_min, 2),
                 "weight_gbs": round(wbytes / (us * 1e-6) / 1e9, 1)}
        if nvec > 1:
            wv = rows * n * nvec
            entry["weight_vector_products_per_s"] = round(wv / (us * 1e-6), 0)
            entry["roofline"] = {"bound": "alu", "unit": "f32 ops/s",
                                 "achieved": round(wv * CHAIN_OPS_PER_WEIGHT_VECTOR / (us * 1e-6), 0),
                                 "peak": roof,
                                 "frac": round(wv * CHAIN_OPS_PER_WEIGHT_VECTOR / (us * 1e-6) / roof, 4),
                                 "roof": "definition's f32 chain, 5 ops per 16 weight-vector products, on all "
                                         "SMs' f32 lanes at 2070 MHz"}
            by_kernel = {}
            for k in ("dp4a", "tensor"):
                prev = binding.gemm_small_kernel(k)
                try:
                    by_kernel[k] = round(cold_median()[0], 2)
                finally:
                    binding.gemm_small_kernel(prev)
            entry["us_by_kernel"] = by_kernel
        res[name] = entry
        del packed, q, d, out
    del flush
    torch.cuda.empty_cache()
    return res


def time_q2_set(dev, steps: int, layers: int = 32):
    """The same decode set with Q2_0 (ternary) weights, one q2_0_gemv_multi
    launch per step, timed like the headline (graph replays, inputs larger
    than L2)."""
    import torch
    from decode_q1_gemv_gb300 import synth
    from decode_q1_gemv_gb300.decode_set import DecodeSet

    shapes = synth.decode_set_shapes()
    if layers < synth.LLAMA3_8B_LAYERS:
        shapes = shapes[:7 * layers]
    ds = DecodeSet(seed=3, device=str(dev), shapes=shapes, fmt="q2")
    g = ds._capture(lambda: ds.step(schedule="set"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ms = _time_graph(g, steps, torch.cuda.current_stream(dev))
    wb = ds.weight_bytes
    peak, _ = measured_peaks()
    launch_bytes = wb + ds.activation_bytes + ds.output_bytes
    res = {"products": len(ds.shapes), "weight_bytes": wb, "us": round(ms * 1e3, 2),
           "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 2),
           "hbm_frac_of_measured": round(wb / (ms * 1e-3) / 1e9 / peak, 4),
           "roofline_frac": round(launch_bytes / (ms * 1e-3) / 1e9 / peak, 4),
           "kernel": "k_q1_multi<8,256,FmtQ2> (q2_0_gemv_multi)",
           "data": "synthetic ternary: P(-1) = P(+1) = 1/4, P(0) = 1/2; halfnormal fp16 scales"}
    del ds, g
    torch.cuda.empty_cache()
    return res


def run_q2_only(args):
    import torch
    from decode_q1_gemv_gb300 import binding
    binding.load()
    dev = torch.device("cuda:0")
    print(json.dumps({"q2_0_decode_set": time_q2_set(dev, args.steps, args.layers)}), flush=True)
    return 0


def run_configs_only(args):
    import torch

    torch.cuda.set_device(0)
    from decode_q1_gemv_gb300 import binding

    binding.load()
    only = [c for c in args.config.split(",") if c] if args.config else None
    res = time_other_configs(torch.device("cuda", 0), reps=max(args.steps, 1), only=only)
    print(json.dumps({"other_configs_cold_l2": res}), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)

    from decode_q1_gemv_gb300 import binding
    from decode_q1_gemv_gb300.decode_set import DecodeSet

    binding.load()
    from decode_q1_gemv_gb300 import synth
    shapes = synth.decode_set_shapes()
    if args.layers < synth.LLAMA3_8B_LAYERS:
        shapes = shapes[:7 * args.layers]  # a smaller set (profiling runs); the lm_head is dropped too
    ds = DecodeSet(seed=3, device=str(dev), shapes=shapes)
    schedules = ["set"] + [s for s in args.schedules.split(",") if s and s != "set"]
    graphs = {sch: ds._capture(lambda sch=sch: ds.step(schedule=sch)) for sch in schedules}
    graph = graphs["set"]
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def reduce_max(v: float) -> float:
        return max_over_ranks(v, world, dist, dev)

    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()

    # ---- main timed region: K decode steps (one launch each), clocks sampled
    # over a window of the same load around it
    sampler = ClockSampler(local)
    sampler.start()
    t_pre = time.time()
    while time.time() - t_pre < 0.6:
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    step_ms = _time_graph(graph, args.steps, stream)
    barrier()
    t_post = time.time()
    while time.time() - t_post < 0.6:
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize()
    sampler.stop()
    step_ms = reduce_max(step_ms)

    # ---- median and minimum of single replays of the timed step (the value
    # above is the mean over the K bracketed replays)
    singles = []
    for _ in range(max(args.steps // 4, 10)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        singles.append(e0.elapsed_time(e1) * 1e3)
    singles.sort()
    set_median_us, set_min_us = singles[len(singles) // 2], singles[0]

    # ---- the same work under the other schedules (decode-order dependencies)
    sched_us = {"set": round(step_ms * 1e3, 2)}
    for sch in schedules[1:]:
        g = graphs[sch]
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        sched_us[sch] = round(reduce_max(_time_graph(g, max(args.steps // 4, 10), stream)) * 1e3, 2)
    # the dependent schedules without the next launch's L2 prefetch, for comparison
    sched_us_nopf = {}
    ds.prefetch_next = False
    for sch in [s for s in schedules[1:] if s in ("grouped", "decode")]:
        g = ds._capture(lambda sch=sch: ds.step(schedule=sch))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        sched_us_nopf[sch] = round(reduce_max(_time_graph(g, max(args.steps // 4, 10), stream)) * 1e3, 2)
        del g
    ds.prefetch_next = True

    # ---- end to end through the public API with host buffers: the
    # activations and outputs live in pinned host memory, and every step's
    # bytes cross the host link (NVLink-C2C on a GB300) inside the timed region.
    # Three flows: (1) q8_quantize_act reads every activation from the host in
    # one launch into device q/d, then q1_0_gemv_multi writes the outputs to
    # the host (the headline e2e); (2) q1_0_gemv_multi alone on the host
    # activations (zero copy: each product's table build reads them);
    # (3) explicit copies into and out of device buffers around the set launch.
    host_x = ds.x_all.cpu().pin_memory()
    host_out = torch.empty(ds.out_all.shape, dtype=ds.out_all.dtype, pin_memory=True)
    qh_arr = binding.product_array(
        [(ds.packed_view(i), rows, n, None, ds.q[i], ds.d[i], host_out[ds.out_off[i]:ds.out_off[i] + rows])
         for i, (_, rows, n) in enumerate(ds.shapes)])
    zc_arr = binding.product_array(
        [(ds.packed_view(i), rows, n, host_x[ds.x_off[i]:ds.x_off[i] + n], None, None,
          host_out[ds.out_off[i]:ds.out_off[i] + rows]) for i, (_, rows, n) in enumerate(ds.shapes)])

    def quantize_then_multiply():
        binding.quantize(host_x, ds.q_all, ds.d_all)
        binding.gemv_multi(array=qh_arr)

    def time_host_flow(fn):
        g = ds._capture(fn)
        for _ in range(3):
            g.replay()
            stream.synchronize()
        barrier()
        z0, z1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        z0.record(stream)
        for _ in range(args.steps):
            g.replay()
            stream.synchronize()  # the step's result is in host memory
        z1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return reduce_max(z0.elapsed_time(z1) / args.steps)

    qh_ms = time_host_flow(quantize_then_multiply)
    host_outs = [host_out.clone()]
    zc_ms = time_host_flow(lambda: binding.gemv_multi(array=zc_arr))
    host_outs.append(host_out.clone())
    for _ in range(3):
        ds.x_all.copy_(host_x, non_blocking=True)
        graph.replay()
        host_out.copy_(ds.out_all, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.steps):
        ds.x_all.copy_(host_x, non_blocking=True)
        graph.replay()
        host_out.copy_(ds.out_all, non_blocking=True)
        stream.synchronize()  # the step's result is on the host
    x1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = reduce_max(x0.elapsed_time(x1) / args.steps)
    host_outs.append(host_out.clone())
    graph.replay()
    torch.cuda.synchronize()
    set_bits = ds.out_all.cpu().view(torch.int32)
    e2e_identical = all(torch.equal(h.view(torch.int32), set_bits) for h in host_outs)

    other = None
    if rank == 0 and args.configs:
        other = time_other_configs(dev)
    q2 = None
    if rank == 0 and args.q2:
        q2 = time_q2_set(dev, max(args.steps // 2, 20), args.layers)

    wb = ds.weight_bytes
    peak, peak_kind = measured_peaks()
    value = world * wb / (step_ms * 1e-3) / 1e9
    launch_bytes = wb + ds.activation_bytes + ds.output_bytes   # one launch per step
    achieved = launch_bytes / (step_ms * 1e-3) / 1e9
    traffic = recorded_traffic()
    clocks = sampler.summary()

    cpu = ctx = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ds.out_all.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        gpu_out = ds.out_all.cpu().numpy()
        gbs, desc, cores, parity = cpu_oracle_set(ds, gpu_out, threads=os.cpu_count() or 1)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
        ctx = cpu_context()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.layers >= 32 else f"first {args.layers} layers of the set",
                       "products": len(ds.shapes), "batch": 1, "weight_bytes": wb,
                       "schedule": "set: one q1_0_gemv_multi launch, q8_0 quantization fused",
                       "l2": f"inputs larger than L2: each step streams {wb / 1e9:.3f} GB of weights",
                       "parallelism": f"replicas x{world}"},
            "us_per_set": round(step_ms * 1e3, 2),
            "us_per_set_single_replays": {"median": round(set_median_us, 2), "min": round(set_min_us, 2),
                                          "replays": len(singles)},
            "other_configs_cold_l2": other,
            "q2_0_decode_set": q2,
            "hbm_frac_of_measured": round(value / world / peak, 4),
            "us_per_set_by_schedule": sched_us,
            "us_per_set_without_prefetch": sched_us_nopf,
            "launches_by_schedule": {sch: ds.launches(sch) for sch in schedules},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "frac_of_nominal_8000_gbs": round(achieved / 8000.0, 4),
                         "kernel": "k_q1_multi (q1_0_gemv_multi, 225 products)", "launches_per_step": 1,
                         "algorithmic_bytes_per_launch": launch_bytes, "peak_source": peak_kind},
            "e2e": {"value": round(world * wb / (qh_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": int(host_x.numel() * 4), "d2h_bytes_per_step": int(host_out.numel() * 4),
                    "ms_per_step": round(qh_ms, 4), "launches_per_step": 2,
                    "transfer": "q8_quantize_act reads the pinned host activations over the host link into "
                                "device q/d, then q1_0_gemv_multi writes the outputs to pinned host memory; "
                                "then a stream sync"},
            "e2e_zero_copy": {"value": round(world * wb / (zc_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                              "h2d_bytes_per_step": int(host_x.numel() * 4),
                              "d2h_bytes_per_step": int(host_out.numel() * 4), "ms_per_step": round(zc_ms, 4),
                              "launches_per_step": 1,
                              "transfer": "q1_0_gemv_multi on pinned host activations and outputs, read and "
                                          "written by the kernel over the host link; then a stream sync"},
            "e2e_outputs_identical_to_set": e2e_identical,
            "e2e_with_copies": {"value": round(world * wb / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                                "h2d_bytes_per_step": int(host_x.numel() * 4),
                                "d2h_bytes_per_step": int(host_out.numel() * 4), "ms_per_step": round(e2e_ms, 4),
                                "transfer": "cudaMemcpyAsync of the activations in and the outputs out around "
                                            "the launch, then a stream sync"},
            "gpu_launches": ds.launches("set") * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "parity": parity,
            "cpu_context": ctx,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip timing the single-product and batched configurations")
    ap.add_argument("--configs-only", action="store_true",
                    help="time only the single-product and batched configurations (for profiling)")
    ap.add_argument("--config", default="",
                    help="with --configs-only: comma list of configuration names to time (" +
                         ", ".join(c[0] for c in OTHER_CONFIGS) + "); empty for all")
    ap.add_argument("--no-q2", dest="q2", action="store_false",
                    help="skip timing the decode set with Q2_0 (ternary) weights")
    ap.add_argument("--q2-only", action="store_true",
                    help="time only the Q2_0 decode set (for profiling)")
    ap.add_argument("--layers", type=int, default=32, help="layers of the decode set (32 = full set with lm_head)")
    ap.add_argument("--schedules", default="grouped,decode,separate",
                    help="schedules timed besides 'set' (comma list; empty for none)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.configs_only:
        return run_configs_only(args)
    if args.q2_only:
        return run_q2_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
