"""Benchmark of the fused row softmax on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all] [--impl ours|reference]
                    [--op softmax|rmsnorm|layernorm]

One step is one rowsoftmax_fwd call (the whole hot path: load, max, exp,
sum, normalise, store) over one batch of the workload.  With --op rmsnorm or
layernorm a step is one rmsnorm_fwd / layernorm_fwd call (with weight, and
bias for LayerNorm) on the same shapes.  The default workload is the largest
one, bf16 attention scores [16, 32, 2048, 2048] as 1048576 x 2048 rows
(8.59 GB moved per step), timed with the plain rowsoftmax_fwd; the line also
carries, under "all_configs", the device-timed figures of the other four
workloads and of rowsoftmax_causal_fwd on the same scores from the same run.  Rank 0 prints one JSON line per
workload with achieved HBM GB/s (bytes = M * N * (in + out element size)),
rows/s, the roofline fraction of the kernel against the measured HBM copy
bandwidth, the end-to-end figure through the C ABI with host buffers, the
SM clocks sampled during the timed region, and the CPU oracle timed on a
bounded sample of the same workload on the host cores.

Under torchrun every rank runs the same workload on its own GPU (replicas,
weak scaling, no collective on the data path); the timed region is bracketed
by barriers and the max over ranks is taken.
"""
from __future__ import annotations

import argparse
import csv
import ctypes
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "bf16_causal_16x32x2048"
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
CSRC = os.path.join(ROOT, "memory_bound_row_gb300", "csrc")


# Sources outside the kernels the benchmark lines time (the split-row kernels
# have their own translation unit and their own --split measurements).
TRAFFIC_HASH_EXCLUDES = ("rs_split.cu",)


def kernel_source_hash() -> str:
    """Hash of the CUDA/C++ sources of the library behind the benchmark lines
    (every source but TRAFFIC_HASH_EXCLUDES): a committed ncu traffic figure is
    only reported while the sources it was taken on are unchanged."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in TRAFFIC_HASH_EXCLUDES:
            with open(os.path.join(CSRC, f), "rb") as fh:
                h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu capture, or None when
    there is none or the kernel sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    ent = data.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def finish(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for rec in csv.reader(io.StringIO(out)):
            if len(rec) < 10:
                continue
            rec = [r.strip() for r in rec]
            try:
                ts = time.mktime(time.strptime(rec[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + rec[0].split(".")[1]) if "." in rec[0] else 0.0
                rows.append((ts, float(rec[2]), float(rec[3]), rec[5:]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside or rows
        if not use:
            return None
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, val in zip(names, r[3][1:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_region": len(inside)}


def max_over_ranks(x: float, device) -> float:
    """The max of x over all ranks of the process group (x itself without one)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_step: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processed `steps` steps of its own
    replica of the workload in at most max_ms milliseconds."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


OP_CODES = {"softmax": 0, "rmsnorm": 1, "layernorm": 2}
OP_EPS = {"softmax": 0.0, "rmsnorm": 1e-6, "layernorm": 1e-5}
OP_METRIC = {"softmax": "achieved HBM GB/s (row softmax)", "rmsnorm": "achieved HBM GB/s (RMSNorm)",
             "layernorm": "achieved HBM GB/s (LayerNorm)"}


def op_workload(op: str, name: str):
    from memory_bound_row_gb300 import workloads as W

    return W.WORKLOADS[name] if op == "softmax" else W.norm_workload(name)


def op_bytes(op: str, w) -> int:
    """Algorithmic bytes of one call: every element read once and written
    once, plus the weight (and bias) vector read once."""
    vectors = {"softmax": 0, "rmsnorm": 1, "layernorm": 2}[op]
    return w.algorithmic_bytes + vectors * w.N * w.elem_size


def traffic_key(op: str, name: str, causal: bool = False) -> str:
    if op == "softmax":
        return f"causal:{name}" if causal else name
    return f"{op}:{name}"


def oracle_op(op: str, x_np, fmt: str, n_cols: int, params, threads: int, out=None):
    """The oracle's result for the rows of x_np, on `threads` host threads."""
    import concurrent.futures as cf

    import numpy as np

    import oracle

    if op == "softmax":
        return oracle.softmax_store(x_np, fmt, n_cols, nthreads=threads, out=out)
    w, b = params
    blocks = [blk for blk in np.array_split(np.arange(x_np.shape[0]), threads) if len(blk)]

    def work(blk):
        part = x_np[blk[0]: blk[-1] + 1]
        if op == "rmsnorm":
            return oracle.rmsnorm_f64(part, fmt, w, OP_EPS[op], n_cols)
        return oracle.layernorm_f64(part, fmt, w, b, OP_EPS[op], n_cols)

    with cf.ThreadPoolExecutor(len(blocks)) as ex:
        return list(ex.map(work, blocks))


def host_params(w):
    """The weight and bias vectors of workload w in the oracle's storage format."""
    import numpy as np
    import torch

    from memory_bound_row_gb300 import workloads as W

    wt, bs = W.norm_params(w.N, w.dtype, w.seed, "cpu")
    conv = (lambda t: t.view(torch.int16).numpy().view(np.uint16)) if w.dtype == "bf16" else (lambda t: t.numpy())
    return conv(wt), conv(bs)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, workloads):
    """The CPU oracle timed on the host cores: each step is the oracle over a
    bounded sample of rows of the workload (rank 0 only)."""
    import numpy as np
    import torch

    import oracle
    from memory_bound_row_gb300 import workloads as W

    world, rank, _ = dist_setup()
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    op = args.op
    for name in workloads:
        w = op_workload(op, name)
        fmt = w.dtype
        params = host_params(w) if op != "softmax" else None
        # A probe of up to 1024 rows sizes the per-step sample: about a minute of
        # oracle time for the whole run, at most 65536 rows a step.
        probe_rows = min(w.M, 1024)
        store = lambda t: t.view(torch.int16).numpy().view(np.uint16) if fmt == "bf16" else t.numpy()
        x_np = store(W.generate(w, "cpu", 0, probe_rows)[:, : w.N].contiguous())
        oracle_op(op, x_np[: min(probe_rows, cores)], fmt, w.N, params, cores)  # first call: loads the oracle
        t = time.perf_counter()
        oracle_op(op, x_np, fmt, w.N, params, cores)
        per_row = (time.perf_counter() - t) / probe_rows
        budget = 60.0  # seconds for the whole run
        rows_per_step = max(1, min(w.M, 65536, int(budget / max(1, args.steps + args.warmup) / per_row)))
        if rows_per_step > probe_rows:
            x_np = store(W.generate(w, "cpu", 0, rows_per_step)[:, : w.N].contiguous())
        sample = x_np[:rows_per_step]
        for _ in range(args.warmup):
            oracle_op(op, sample, fmt, w.N, params, cores)
        t = time.perf_counter()
        for _ in range(args.steps):
            oracle_op(op, sample, fmt, w.N, params, cores)
        dt = (time.perf_counter() - t) / args.steps
        nbytes = rows_per_step * w.N * 2 * w.elem_size
        gbs = nbytes / dt / 1e9
        sample_desc = f"{rows_per_step} of {w.M} rows per step ({w.description}), host oracle, fp64"
        line = {
            "impl": "reference", "metric": OP_METRIC[op], "value": round(gbs, 4),
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "rows_per_s": round(rows_per_step / dt, 2),
            "config": {"workload": name, "op": op, "M": w.M, "N": w.N, "row_stride": w.ld, "storage": w.dtype,
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample_desc},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)


def cpu_baseline(w, x_dev, op: str = "softmax", seconds: float = 3.0) -> dict:
    """The oracle, as it stands, on a bounded sample of rows of the workload
    on all host cores, repeated for about `seconds` of wall time."""
    import numpy as np
    import torch

    cores = os.cpu_count() or 1
    fmt = w.dtype
    params = host_params(w) if op != "softmax" else None

    def host(rows):
        t = x_dev[:rows, : w.N].cpu().contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if fmt == "bf16" else t.numpy()

    probe = min(w.M, max(cores, 16))
    xs = host(probe)
    t = time.perf_counter()
    oracle_op(op, xs, fmt, w.N, params, cores)
    per_row = (time.perf_counter() - t) / probe
    rows = int(min(w.M, max(probe, seconds / 4 / max(per_row, 1e-9))))
    xs = host(rows)
    out = np.zeros_like(xs)
    passes = 0
    t = time.perf_counter()
    while True:
        oracle_op(op, xs, fmt, w.N, params, cores, out=out)
        passes += 1
        if time.perf_counter() - t >= seconds:
            break
    dt = (time.perf_counter() - t) / passes
    nbytes = rows * w.N * 2 * w.elem_size
    # The same oracle on one thread, over the first rows of the sample,
    # repeated for about a third of `seconds`.
    rows1 = max(1, rows // cores)
    passes1 = 0
    t = time.perf_counter()
    while True:
        oracle_op(op, xs[:rows1], fmt, w.N, params, 1, out=out[:rows1])
        passes1 += 1
        if time.perf_counter() - t >= seconds / 3:
            break
    dt1 = (time.perf_counter() - t) / passes1
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {w.M} rows x {passes} passes, fp64 {op} oracle"
                      f"{' writing ' + w.dtype if op == 'softmax' else ''}, "
                      f"{dt * passes:.1f} s wall on {cores} threads",
            "rows_per_s": round(rows / dt, 2),
            "single_thread": {"value": round(rows1 * w.N * 2 * w.elem_size / dt1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"first {rows1} rows x {passes1} passes, {dt1 * passes1:.1f} s on 1 thread"}}


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e bandwidth as specified (nominal, not measured)


def pick_graph_launches(steps: int, nsets: int, est_ms: float) -> int:
    """Launches per CUDA graph: the largest divisor of `steps` (at most 64)
    whose replay holds about a millisecond of work or less, so that long
    kernels get several replays for the per-replay median while short ones
    are not stretched by host launch cost; a multiple of the rotating buffer
    sets where one qualifies."""
    divisors = [g for g in range(1, min(64, steps) + 1) if steps % g == 0]
    fit = [g for g in divisors if g == 1 or g * est_ms <= 1.0]
    pref = [g for g in fit if g % nsets == 0]
    return max(pref or fit)


def measure(args, name, ctx, full: bool, causal_summary: bool = False):
    """Times K graph-replayed launches of the row operation on workload
    `name`.  Returns the JSON line (rank 0; None elsewhere).  With full=False
    only the device-timed figures are taken (no end-to-end leg, clocks or CPU
    baseline): the compact per-workload summary of the headline line."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import memory_bound_row_gb300 as rs
    from memory_bound_row_gb300 import workloads as W

    lib, dev, world, rank, local, peak, peak_src, opts = (ctx[k] for k in (
        "lib", "dev", "world", "rank", "local", "peak", "peak_src", "opts"))
    op = args.op
    causal = (args.causal and full) or causal_summary
    w = op_workload(op, name)
    if args.rows and full:
        w = W.Workload(w.name, w.dtype, min(args.rows, w.M), w.N, w.ld, w.seed, w.kind,
                       f"first {min(args.rows, w.M)} rows of: {w.description}")
    code = {"f32": rs.RS_F32, "f16": rs.RS_F16, "bf16": rs.RS_BF16}[w.dtype]
    set_bytes = 2 * w.M * w.ld * w.elem_size
    nsets = max(1, math.ceil(4 * L2_BYTES / set_bytes))
    xs = [W.generate(w, dev) for _ in range(1)]
    xs += [xs[0].clone() for _ in range(nsets - 1)]
    ys = [torch.empty_like(xs[0]) for _ in range(nsets)]
    stream = torch.cuda.current_stream(dev)
    s_handle = ctypes.c_void_p(stream.cuda_stream)
    args_list = [(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr())) for x, y in zip(xs, ys)]
    wt = bs = None
    if op != "softmax":
        wt, bs = W.norm_params(w.N, w.dtype, w.seed, dev)
        p_w = ctypes.c_void_p(wt.data_ptr())
        p_b = ctypes.c_void_p(bs.data_ptr()) if op == "layernorm" else None

    def call(a, b, st):
        if op == "softmax" and causal:
            return lib.rowsoftmax_causal_fwd_ex(a, b, w.M, w.N, w.ld, w.ld, w.N, 0, code, st, opts)
        if op == "softmax":
            return lib.rowsoftmax_fwd_ex(a, b, w.M, w.N, w.ld, w.ld, code, st, opts)
        return lib.rownorm_fwd_ex(OP_CODES[op], a, b, p_w, p_b, w.M, w.N, w.ld, w.ld, OP_EPS[op], code, st, opts)

    def step(i, st=None):
        a, b = args_list[i % nsets]
        rc = call(a, b, st if st is not None else s_handle)
        if rc != rs.RS_OK:
            raise rs.RowSoftmaxError(rc, rs.rowsoftmax_last_cuda_error())

    # Warm-up launches, launched directly; their average (an upper bound of
    # the kernel's time) sizes the graphs below.
    warm = max(3, args.warmup)
    step(0)
    torch.cuda.synchronize()
    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for i in range(1, warm):
        step(i)
    w1.record(stream)
    torch.cuda.synchronize()
    est_ms = w0.elapsed_time(w1) / max(1, warm - 1)

    # The K timed steps are replayed from a CUDA graph of G consecutive
    # launches (pick_graph_launches), so host launch cost does not stretch
    # short kernels; the graph is replayed once untimed before the events
    # (its first replay carries the upload), then K / G times inside them.
    G = pick_graph_launches(args.steps, nsets, est_ms)
    reuse_mb = min(G, nsets) * set_bytes / 1e6  # bytes of other sets between two uses of one set
    graph_stream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(graph_stream):
        g_handle = ctypes.c_void_p(graph_stream.cuda_stream)
        for i in range(G):  # same buffers as the capture, outside it
            step(i, g_handle)
        graph_stream.synchronize()
        with torch.cuda.graph(graph, stream=graph_stream, capture_error_mode="relaxed"):
            for i in range(G):
                step(i, g_handle)
        graph.replay()  # untimed: the first replay of a fresh graph
    torch.cuda.synchronize()
    replays = args.steps // G
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if (rank == 0 and full) else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    # One event between replays as well: the median over the replays is
    # reported beside the whole region's figure (the events add no work).
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    with torch.cuda.stream(graph_stream):  # replay() launches on the current stream
        e_start.record(graph_stream)
        marks[0].record(graph_stream)
        for i in range(replays):
            graph.replay()
            marks[i + 1].record(graph_stream)
        e_end.record(graph_stream)
    torch.cuda.synchronize()
    per_replay = sorted(marks[i].elapsed_time(marks[i + 1]) / G for i in range(replays))
    if sampler:
        sampler.mark_end()
    if world > 1:
        dist.barrier()
    total_ms = e_start.elapsed_time(e_end)
    # Every step is exactly one launch of the library's kernel, back to back
    # on graph_stream: the average launch duration is total / K.
    kern_ms = total_ms / args.steps
    total_ms = max_over_ranks(total_ms, dev)
    clocks = sampler.finish() if sampler else None

    # Context for the roofline: a plain device-to-device copy of the same
    # buffer sets (torch copy_, whole buffers, padding included), timed over
    # K steps on the same box right after the kernel, both replayed from a
    # CUDA graph as the kernel is and launched directly as the measured peak
    # was; the faster counts.  (Each way has sizes where it measured far below
    # the other: graph-captured copies of 512 MB and more at half the
    # bandwidth, direct launches of ~50 us copies about 5 % low.)
    def time_copies(use_graph):
        if use_graph:
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.stream(graph_stream):
                for i in range(G):
                    ys[i % nsets].copy_(xs[i % nsets])
                graph_stream.synchronize()
                with torch.cuda.graph(cg, stream=graph_stream, capture_error_mode="relaxed"):
                    for i in range(G):
                        ys[i % nsets].copy_(xs[i % nsets])
                cg.replay()
        else:
            with torch.cuda.stream(graph_stream):
                for i in range(3):
                    ys[i % nsets].copy_(xs[i % nsets])
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(graph_stream):
            c0.record(graph_stream)
            if use_graph:
                for _ in range(replays):
                    cg.replay()
            else:
                for i in range(args.steps):
                    ys[i % nsets].copy_(xs[i % nsets])
            c1.record(graph_stream)
        torch.cuda.synchronize()
        return (set_bytes * args.steps) / (c0.elapsed_time(c1) * 1e-3) / 1e9

    copy_gbs = max(time_copies(True), time_copies(False))

    ms_per_step = total_ms / args.steps
    nbytes = op_bytes(op, w)
    full_bytes = nbytes
    if causal:
        # The mask's line counts the least traffic it allows -- kept elements
        # read, every element written -- the bytes the kernel must move; the
        # plain softmax's M x N x (in + out) bytes are given beside it.
        kept = int(np.minimum(np.arange(w.M, dtype=np.int64) % w.N + 1, w.N).sum())
        nbytes = (kept + w.M * w.N) * w.elem_size
    value = job_gbs(world, nbytes, args.steps, total_ms)
    achieved = nbytes / (kern_ms * 1e-3) / 1e9

    e2e = None
    if full:
        # End to end through the C ABI with host buffers: every step copies
        # its input in from pinned host memory, runs the call and copies the
        # output back.  Two device buffer pairs let step i+1's copy-in overlap
        # step i's kernel and copy-out (three streams, ordered by events).
        h_in = xs[0].cpu().pin_memory()
        h_out = [torch.empty_like(h_in).pin_memory() for _ in range(2)]
        d_in = [xs[0], xs[1] if nsets > 1 else torch.empty_like(xs[0])]
        d_out = [ys[0], ys[1] if nsets > 1 else torch.empty_like(ys[0])]
        s_in, s_k, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        k_handle = ctypes.c_void_p(s_k.cuda_stream)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_k = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in ev_k + ev_out:
            e.record(torch.cuda.current_stream(dev))

        def e2e_step(i):
            b = i % 2
            s_in.wait_event(ev_k[b])
            with torch.cuda.stream(s_in):
                d_in[b].copy_(h_in, non_blocking=True)
            ev_in[b].record(s_in)
            s_k.wait_event(ev_in[b])
            s_k.wait_event(ev_out[b])
            rc = call(ctypes.c_void_p(d_in[b].data_ptr()), ctypes.c_void_p(d_out[b].data_ptr()), k_handle)
            if rc != rs.RS_OK:
                raise rs.RowSoftmaxError(rc, rs.rowsoftmax_last_cuda_error())
            ev_k[b].record(s_k)
            s_out.wait_event(ev_k[b])
            with torch.cuda.stream(s_out):
                h_out[b].copy_(d_out[b], non_blocking=True)
            ev_out[b].record(s_out)

        e2e_steps = max(4, min(args.steps, 20))
        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_k)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
        e2e = {"value": round(job_gbs(world, nbytes, 1, e2e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": h_in.numel() * h_in.element_size(),
               "d2h_bytes_per_step": h_out[0].numel() * h_out[0].element_size(),
               "ms_per_step": round(e2e_ms, 4),
               "how": f"pinned host input copied in, "
                      f"{('rowsoftmax_causal_fwd' if causal else 'rowsoftmax_fwd') if op == 'softmax' else op + '_fwd'}, "
                      "output copied back, every step; two buffer pairs overlap step i+1's copy-in with step i"}
        del h_in, h_out, d_in, d_out

    rc, flags = rs.rowsoftmax_device_status()
    if rc != rs.RS_OK or flags:
        raise RuntimeError(f"device status word {flags:#x} after the run")

    line = None
    if rank == 0:
        rc, info = rs.rowsoftmax_device_info()
        if op == "softmax" and causal:
            rc, plan = rs.rowsoftmax_causal_plan(xs[0].data_ptr(), ys[0].data_ptr(), w.M, w.N, w.ld, w.ld, w.N,
                                                 0, code, args.options, info)
        elif op == "softmax":
            rc, plan = rs.rowsoftmax_plan(xs[0].data_ptr(), ys[0].data_ptr(), w.M, w.N, w.ld, w.ld, code,
                                          args.options, info)
        else:
            rc, plan = rs.rownorm_plan(OP_CODES[op], xs[0].data_ptr(), ys[0].data_ptr(), wt.data_ptr(),
                                       bs.data_ptr() if op == "layernorm" else None, w.M, w.N, w.ld, w.ld,
                                       OP_EPS[op], code, args.options, info)
        repeats = {"n": replays, "launches_each": G,
                   "median_ms_per_step": round(per_replay[len(per_replay) // 2], 5),
                   "min_ms_per_step": round(per_replay[0], 5),
                   "max_ms_per_step": round(per_replay[-1], 5)}
        if not full:
            line = {"workload": name + (" (rowsoftmax_causal_fwd)" if causal else ""), "value": round(value, 2),
                    "unit": "GB/s", "ms_per_step": round(ms_per_step, 5),
                    "rows_per_s": round(world * w.M / (ms_per_step * 1e-3), 1), "frac": round(achieved / peak, 4),
                    "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                    "frac_of_same_run_copy": round(achieved / copy_gbs, 4), "same_run_copy_gbs": round(copy_gbs, 1),
                    "kernel": rs.PATH_NAMES[plan["path"]], "bytes_per_step": nbytes, "steps": args.steps,
                    "repeats": repeats}
            if causal:  # value and frac count the least traffic the mask allows; the plain count beside it
                line["bytes_counted"] = "kept elements read + all elements written"
                line["full_bytes_per_step"] = full_bytes
                line["full_bytes_gbs"] = round(job_gbs(world, full_bytes, args.steps, total_ms), 2)
        else:
            line = {
                "metric": OP_METRIC[op], "value": round(value, 2), "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
                "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "rows_per_s": round(world * w.M / (ms_per_step * 1e-3), 1),
                "hbm_roofline_frac": round(value / world / peak, 4),
                "hbm_nominal_frac": round(value / world / NOMINAL_HBM_GBS, 4),
                "config": {"workload": name if not args.rows else f"{name} (first {w.M} rows)", "op": op,
                           "M": w.M, "N": w.N, "row_stride": w.ld, "storage": w.dtype,
                           "options": args.options,
                           "bytes_per_step": nbytes, "parallelism": "replicas",
                           "l2": f"{nsets} rotating input/output sets of {set_bytes / 1e6:.0f} MB; "
                                 f"{reuse_mb:.0f} MB pass between two uses of a set (L2 is 129 MB)",
                           "kernel": rs.PATH_NAMES[plan["path"]], "plan": plan},
                "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                             "frac": round(achieved / peak, 4),
                             "traffic": None if (args.options or args.rows)
                             else ncu_traffic(traffic_key(op, name, causal)),
                             "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"
                             if peak_src == "measured" else "fallback 6.8 TB/s",
                             "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                             "nominal_peak": NOMINAL_HBM_GBS,
                             "nominal_source": "GB300 HBM3e bandwidth as specified, 7.9 TB/s (not measured)",
                             "kernel_ms": round(kern_ms, 5),
                             "same_run_copy_gbs": round(copy_gbs, 1),
                             "frac_of_same_run_copy": round(achieved / copy_gbs, 4),
                             "same_run_copy": "torch copy_ of the same rotating buffer sets (padding included), K "
                                              "steps timed right after, the faster of graph-replayed and "
                                              "directly launched"},
                "e2e": e2e,
                "gpu_launches": args.steps,
                **({"causal": {"period": w.N, "diag_offset": 0,
                               "value_counts": "the least traffic the mask allows: kept elements read, all "
                                               "elements written (config.bytes_per_step)",
                               "full_bytes_per_step": full_bytes,
                               "full_bytes_gbs": round(job_gbs(world, full_bytes, args.steps, total_ms), 2),
                               "how": "rowsoftmax_causal_fwd: row r keeps (r mod N) + 1 elements, the masked part "
                                      "is not used and is written as 0"}} if causal else {}),
                "timing": f"{replays} replays of a CUDA graph of {G} launches after one untimed replay; one event "
                          "pair around all of them (value, ms_per_step) and one between consecutive replays "
                          "(repeats)",
                "repeats": repeats,
                "clocks": clocks,
            }
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(w, xs[0], op)
    del xs, ys, graph
    torch.cuda.empty_cache()
    return line


def run_ours(args, workloads):
    import torch
    import torch.distributed as dist

    import memory_bound_row_gb300 as rs
    from memory_bound_row_gb300 import workloads as W

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    peak, peak_src = measured_peaks()
    ctx = {"lib": rs._abi.load(), "dev": dev, "world": world, "rank": rank, "local": local, "peak": peak,
           "peak_src": peak_src, "opts": rs._abi._opts(args.options)}
    for name in workloads:
        # The other workloads first (device-timed only), so that the headline
        # line carries every workload's figure from the same run.
        others = []
        if args.summary_all:
            for other in W.ORDER:
                if other != name:
                    others.append(measure(args, other, ctx, full=False))
            if args.op == "softmax" and "causal" in W.WORKLOADS[name].kind:
                # the mask-aware softmax on the same scores (never reads the masked part)
                others.append(measure(args, name, ctx, full=False, causal_summary=True))
        line = measure(args, name, ctx, full=True)
        if rank == 0:
            if others:
                line["all_configs"] = others
            print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()

SWEEP_CONFIGS = {
    # name: rs_options (None: the planner's choice).  grid_limit -1 means "one
    # wave of resident CTAs" and is resolved per shape.
    "auto": None,
    "rows, one CTA per row group": {"path": 1},
    "rows, persistent": {"path": 1, "grid_limit": -1},
    "ring (bulk copies, persistent)": {"path": 4},
    "rows, 128-thread CTAs": {"path": 1, "block_threads": 128},
    "rows, 256-thread CTAs": {"path": 1, "block_threads": 256},
}


def run_sweep_n(args):
    """The N sweep of the Hugging Face skill page's benchmark harness (fp32
    randn, M = 4096, N = 128 i for i = 2..99) on this library: every point of
    every configuration is first checked (finite, row sums 1 within 1e-5, and
    equal to the planner's configuration within 1e-6 element-wise; the
    configurations themselves are covered by the parity tests), then timed as
    graph-replayed back-to-back launches over rotating buffers (more than 4x
    L2 between two uses of a buffer).  One JSON line per (N, configuration)."""
    import torch

    import memory_bound_row_gb300 as rs
    from memory_bound_row_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = rs._abi.load()
    peak, _ = measured_peaks()
    rc, info = rs.rowsoftmax_device_info()
    M = 4096
    for i in range(2, 100):
        N = 128 * i
        w = W.custom(M, N, "f32", seed=0, kind="normal1")
        x0 = W.generate(w, dev)
        set_bytes = 2 * M * N * 4
        nsets = max(1, math.ceil(4 * L2_BYTES / set_bytes))
        xs = [x0] + [x0.clone() for _ in range(nsets - 1)]
        ys = [torch.empty_like(x0) for _ in range(nsets)]
        torch.cuda.synchronize()  # the inputs are made on torch's stream; the timed calls run on their own
        first = None
        for name, opts in SWEEP_CONFIGS.items():
            o = dict(opts) if opts else None
            if o and o.get("grid_limit") == -1:
                o["grid_limit"] = 0
                rc, plan = rs.rowsoftmax_plan(xs[0].data_ptr(), ys[0].data_ptr(), M, N, N, N, rs.RS_F32, o, info)
                if rc != rs.RS_OK:
                    continue
                per_sm = max(1, info.max_threads_per_sm // plan["block_threads"])
                o["grid_limit"] = info.sm_count * per_sm
            rc, plan = rs.rowsoftmax_plan(xs[0].data_ptr(), ys[0].data_ptr(), M, N, N, N, rs.RS_F32, o, info)
            if rc != rs.RS_OK:
                continue
            copts = rs._abi._opts(o)
            stream = torch.cuda.Stream(dev)
            h = stream.cuda_stream

            def call(k):
                r = lib.rowsoftmax_fwd_ex(xs[k % nsets].data_ptr(), ys[k % nsets].data_ptr(), M, N, N, N,
                                          rs.RS_F32, h, copts)
                if r != rs.RS_OK:
                    raise rs.RowSoftmaxError(r, rs.rowsoftmax_last_cuda_error())

            with torch.cuda.stream(stream):
                call(0)
            stream.synchronize()
            y = ys[0].double()
            sums_err = float((y.sum(dim=1) - 1.0).abs().max())
            err = 0.0 if first is None else float((y - first).abs().max())
            if first is None:
                first = y.clone()
            if not (bool(torch.isfinite(y).all()) and sums_err <= 1e-5 and err <= 1e-6):
                raise AssertionError(f"N={N} {name}: row sums off by {sums_err:.3e}, {err:.3e} from the planner's")
            G = 20
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                for k in range(G):
                    call(k)
                stream.synchronize()
                with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
                    for k in range(G):
                        call(k)
            torch.cuda.synchronize()
            reps = max(3, args.steps // G)
            with torch.cuda.stream(stream):
                graph.replay()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / (reps * G)
            gbs = 2 * M * N * 4 / (ms * 1e-3) / 1e9
            print(json.dumps({"sweep": "fp32 M=4096 N=128i", "N": N, "config": name, "kernel": rs.PATH_NAMES[plan["path"]],
                              "grid": plan["grid"], "block": plan["block_threads"], "us": round(ms * 1e3, 3),
                              "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "max_rowsum_err": sums_err}), flush=True)
            del graph
        del xs, ys, first
        torch.cuda.empty_cache()


WIDE_SWEEP_N = [256, 512, 768, 1024, 1280, 1536, 2048, 2560, 3072, 3584, 4096, 4608, 5120, 5632, 6144, 8192, 12288,
                16384, 20480, 24576, 28672, 32768, 40960, 49152, 65536]
# "ring4": the ring at 4 units a thread, the shape planned before the measured
# shapes of the planner (rs_options forcing the units a thread).
WIDE_SWEEP_CONFIGS = {"auto": None, "ring": {"path": 4}, "ring4": {"path": 4, "vec_per_thread": 4},
                      "cluster": {"path": 2}}


def run_sweep_wide(args):
    """16-bit rows of 256..65536 values (M = 2^28 / N: 512 MB a tensor) for
    the --op row operation, through the planner's choice, the bulk-copy ring
    (the planner's ring shape, and at 4 units a thread) and the
    register-holding clusters, where each has a plan; with --causal, the
    softmax under a causal mask of period N (row r keeps r mod N + 1 values;
    GB/s then count the kept values read and all values written).  Every
    point is checked first on 16 sampled rows against the operation evaluated
    by torch in fp64 on the decoded inputs (softmax also: row sums within
    1e-2), and the configurations against each other; then timed as
    graph-replayed launches over rotating buffers.  One JSON line per (N,
    configuration)."""
    import numpy as np
    import torch

    import memory_bound_row_gb300 as rs
    from memory_bound_row_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = rs._abi.load()
    peak, _ = measured_peaks()
    rc, info = rs.rowsoftmax_device_info()
    op, dt = args.op, args.sweep_dtype
    causal = args.causal and op == "softmax"
    code = {"f16": rs.RS_F16, "bf16": rs.RS_BF16}[dt]
    tol = {"f16": 2.0 ** -9, "bf16": 2.0 ** -6}[dt]  # a few units in the last place of the output
    widths = [int(v) for v in args.widths.split(",")] if getattr(args, "widths", None) else WIDE_SWEEP_N
    for N in widths:
        M = (1 << 28) // N
        w = W.custom(M, N, dt, seed=5, kind="offset50" if op == "layernorm" else "normal1")
        x0 = W.generate(w, dev)
        wt, bs = W.norm_params(N, dt, 5, dev)
        set_bytes = 2 * M * N * 2
        nsets = max(1, math.ceil(4 * L2_BYTES / set_bytes))
        xs = [x0] + [x0.clone() for _ in range(nsets - 1)]
        ys = [torch.empty_like(x0) for _ in range(nsets)]
        rows = torch.linspace(0, M - 1, 16, device=dev).long()
        xr = x0[rows].double()
        if causal:  # row r keeps its first r mod N + 1 values, the rest is 0
            keep = (rows % N + 1)[:, None]
            cols = torch.arange(N, device=dev)[None, :]
            ref = torch.softmax(xr.masked_fill(cols >= keep, -math.inf), dim=1)
        elif op == "softmax":
            ref = torch.softmax(xr, dim=1)
        elif op == "rmsnorm":
            ref = xr * torch.rsqrt((xr * xr).mean(dim=1, keepdim=True) + OP_EPS[op]) * wt.double()
        else:
            mu = xr.mean(dim=1, keepdim=True)
            ref = (xr - mu) * torch.rsqrt(((xr - mu) ** 2).mean(dim=1, keepdim=True) + OP_EPS[op]) * wt.double() \
                + bs.double()
        torch.cuda.synchronize()
        first = None
        for name, opts in WIDE_SWEEP_CONFIGS.items():
            copts = rs._abi._opts(opts)
            if causal:
                rc, plan = rs.rowsoftmax_causal_plan(xs[0].data_ptr(), ys[0].data_ptr(), M, N, N, N, N, 0, code,
                                                     opts, info)
            elif op == "softmax":
                rc, plan = rs.rowsoftmax_plan(xs[0].data_ptr(), ys[0].data_ptr(), M, N, N, N, code, opts, info)
            else:
                rc, plan = rs.rownorm_plan(OP_CODES[op], xs[0].data_ptr(), ys[0].data_ptr(), wt.data_ptr(),
                                           bs.data_ptr() if op == "layernorm" else None, M, N, N, N, OP_EPS[op],
                                           code, opts, info)
            if rc != rs.RS_OK:
                continue
            stream = torch.cuda.Stream(dev)
            h = stream.cuda_stream
            pb = bs.data_ptr() if op == "layernorm" else None

            def call(k):
                if causal:
                    r = lib.rowsoftmax_causal_fwd_ex(xs[k % nsets].data_ptr(), ys[k % nsets].data_ptr(), M, N, N, N,
                                                     N, 0, code, h, copts)
                elif op == "softmax":
                    r = lib.rowsoftmax_fwd_ex(xs[k % nsets].data_ptr(), ys[k % nsets].data_ptr(), M, N, N, N, code,
                                              h, copts)
                else:
                    r = lib.rownorm_fwd_ex(OP_CODES[op], xs[k % nsets].data_ptr(), ys[k % nsets].data_ptr(),
                                           wt.data_ptr(), pb, M, N, N, N, OP_EPS[op], code, h, copts)
                if r != rs.RS_OK:
                    raise rs.RowSoftmaxError(r, rs.rowsoftmax_last_cuda_error())

            with torch.cuda.stream(stream):
                call(0)
            stream.synchronize()
            y = ys[0][rows].double()
            err = float(((y - ref).abs() / (1.0 + ref.abs())).max())
            agree = 0.0 if first is None else float(((y - first).abs() / (1.0 + first.abs())).max())
            if first is None:
                first = y.clone()
            sums = float((y.sum(dim=1) - 1.0).abs().max()) if op == "softmax" else 0.0
            if not (bool(torch.isfinite(y).all()) and err <= tol and agree <= 2 * tol and sums <= 1e-2):
                raise AssertionError(f"{op} N={N} {name}: error {err:.3e}, {agree:.3e} from the planner's")
            G = 20
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                for k in range(G):
                    call(k)
                stream.synchronize()
                with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
                    for k in range(G):
                        call(k)
            torch.cuda.synchronize()
            reps = max(3, args.steps // G)
            with torch.cuda.stream(stream):
                graph.replay()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / (reps * G)
            nbytes = 2 * M * N * 2 + {"softmax": 0, "rmsnorm": 1, "layernorm": 2}[op] * N * 2
            if causal:  # kept values read, all written
                kept = int(np.minimum(np.arange(M, dtype=np.int64) % N + 1, N).sum())
                nbytes = (kept + M * N) * 2
            gbs = nbytes / (ms * 1e-3) / 1e9
            print(json.dumps({"sweep": f"{dt} rows, M = 2^28 / N" + (", causal mask of period N" if causal else ""),
                              "op": op, "N": N, "M": M, "config": name,
                              "kernel": rs.PATH_NAMES[plan["path"]], "cluster": plan["cluster_size"],
                              "threads": plan["block_threads"], "threads_per_row": plan["threads_per_row"],
                              "units_a_thread": plan["vec_per_thread"], "stages": plan["stages"],
                              "grid": plan["grid"], "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                              "frac": round(gbs / peak, 4), "max_rel_err": round(err, 6)}), flush=True)
            del graph
        del xs, ys, first
        torch.cuda.empty_cache()


SPLIT_SHAPES = [(1, 1 << 26, "f16"), (4, 1 << 22, "bf16"), (16, 1 << 20, "f16"), (64, 1 << 18, "bf16"),
                (512, 131072, "f16")]


def graph_ms(call, steps: int, stream) -> float:
    """Milliseconds per call: `steps` calls replayed from one CUDA graph,
    after one untimed replay, between CUDA events on `stream`."""
    import torch

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for k in range(steps):
            call(k)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
            for k in range(steps):
                call(k)
        graph.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_split(args):
    """The split-row softmax measured on one device (one JSON line each):
    (1) rowsoftmax_split_fwd against rowsoftmax_fwd on few, very wide rows
    (M x N below; GB/s counts M N (in + out) bytes; the split reads x twice);
    (2) the two steps of the vocabulary-parallel softmax on the bf16 causal
    scores split into two column shards of 1024: rowsoftmax_partial_fwd on a
    shard (bytes: its elements read, 8 a row written) and rowsoftmax_finish_fwd
    with both shards' pairs (its elements read and written, the pairs read) or
    with the merged pairs, and rowsoftmax_fwd on the same strided elements.
    Every configuration is first checked against rowsoftmax_fwd on the same
    input (max |difference| within 2^-7 for 16-bit, 1e-6 for fp32); timings
    are graph-replayed launches over rotating buffers (more than 4x L2
    between two uses of a buffer where the tensors are smaller than that)."""
    import torch

    import memory_bound_row_gb300 as rs
    from memory_bound_row_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = rs._abi.load()
    peak, _ = measured_peaks()
    stream = torch.cuda.Stream(dev)
    h = stream.cuda_stream
    steps = max(4, min(args.steps, 64))
    for M, N, dt in SPLIT_SHAPES:
        code = {"f32": rs.RS_F32, "f16": rs.RS_F16, "bf16": rs.RS_BF16}[dt]
        w = W.custom(M, N, dt, seed=9, kind="normal_spike")
        set_bytes = 2 * M * N * w.elem_size
        nsets = max(1, math.ceil(4 * L2_BYTES / set_bytes))
        xs = [W.generate(w, dev)]
        xs += [xs[0].clone() for _ in range(nsets - 1)]
        ys = [torch.empty_like(xs[0]) for _ in range(nsets)]
        rc, need = rs.rowsoftmax_split_workspace_size(M, N, code)
        wss = [torch.empty(max(need, 8), dtype=torch.uint8, device=dev) for _ in range(nsets)]
        ref = rs.softmax(xs[0])
        got = rs.softmax_split(xs[0], workspace=wss[0])
        torch.cuda.synchronize()
        diff = float((ref.double() - got.double()).abs().max())
        if not diff <= (1e-6 if dt == "f32" else 2.0 ** -7):
            raise AssertionError(f"split {M}x{N}: differs from rowsoftmax_fwd by {diff:.3e}")
        del ref, got

        def fwd(k):
            r = lib.rowsoftmax_fwd(xs[k % nsets].data_ptr(), ys[k % nsets].data_ptr(), M, N, N, N, code, h)
            if r != rs.RS_OK:
                raise rs.RowSoftmaxError(r)

        def split(k):
            r = lib.rowsoftmax_split_fwd(xs[k % nsets].data_ptr(), ys[k % nsets].data_ptr(), M, N, N, N, code,
                                         wss[k % nsets].data_ptr(), need, h)
            if r != rs.RS_OK:
                raise rs.RowSoftmaxError(r)

        rc, info = rs.rowsoftmax_device_info()
        rc, plan = rs.rowsoftmax_plan(xs[0].data_ptr(), ys[0].data_ptr(), M, N, N, N, code, None, info)
        nbytes = M * N * 2 * w.elem_size
        for name, fn in (("rowsoftmax_fwd (" + rs.PATH_NAMES[plan["path"]] + ")", fwd), ("rowsoftmax_split_fwd", split)):
            ms = graph_ms(fn, steps, stream)
            gbs = nbytes / (ms * 1e-3) / 1e9
            print(json.dumps({"split": "few wide rows", "M": M, "N": N, "storage": dt, "call": name,
                              "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "max_diff_to_fwd": diff}), flush=True)
        del xs, ys, wss
        torch.cuda.empty_cache()

    # The vocabulary-parallel steps on the bf16 causal scores, two shards.
    wl = W.WORKLOADS["bf16_causal_16x32x2048"]
    M, N, half = wl.M, wl.N, wl.N // 2
    x = W.generate(wl, dev)
    y = torch.empty_like(x)
    pairs = torch.empty((2, M, 2), dtype=torch.float32, device=dev)
    for s in range(2):
        rs.softmax_partial(x[:, s * half:(s + 1) * half], ml=pairs[s])
    for s in range(2):
        rs.softmax_finish(x[:, s * half:(s + 1) * half], pairs, out=y[:, s * half:(s + 1) * half])
    ref = rs.softmax(x)
    torch.cuda.synchronize()
    diff = float((ref.double() - y.double()).abs().max())
    if not diff <= 2.0 ** -7:
        raise AssertionError(f"two shards differ from rowsoftmax_fwd by {diff:.3e}")
    del ref
    code = rs.RS_BF16
    xp = [x[:, 0:half], x[:, half:N]]

    def partial(k):
        r = lib.rowsoftmax_partial_fwd(xp[k % 2].data_ptr(), pairs[k % 2].data_ptr(), M, half, N, code, h)
        if r != rs.RS_OK:
            raise rs.RowSoftmaxError(r)

    def finish(k):
        r = lib.rowsoftmax_finish_fwd(xp[k % 2].data_ptr(), y[:, (k % 2) * half:].data_ptr(), pairs.data_ptr(), 2, M,
                                      half, N, N, code, h)
        if r != rs.RS_OK:
            raise rs.RowSoftmaxError(r)

    merged = rs.softmax_merge(pairs)
    torch.cuda.synchronize()

    def finish1(k):
        r = lib.rowsoftmax_finish_fwd(xp[k % 2].data_ptr(), y[:, (k % 2) * half:].data_ptr(), merged.data_ptr(), 1,
                                      M, half, N, N, code, h)
        if r != rs.RS_OK:
            raise rs.RowSoftmaxError(r)

    def whole(k):  # the row softmax of the same strided elements, for comparison
        r = lib.rowsoftmax_fwd(xp[k % 2].data_ptr(), y[:, (k % 2) * half:].data_ptr(), M, half, N, N, code, h)
        if r != rs.RS_OK:
            raise rs.RowSoftmaxError(r)

    for name, fn, nbytes in (("rowsoftmax_partial_fwd", partial, M * half * 2 + M * 8),
                             ("rowsoftmax_finish_fwd (R = 2)", finish, M * half * 4 + 2 * M * 8),
                             ("rowsoftmax_finish_fwd (R = 1, merged pairs)", finish1, M * half * 4 + M * 8),
                             ("rowsoftmax_fwd on the same shard", whole, M * half * 4)):
        ms = graph_ms(fn, steps, stream)
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({"split": "vocabulary-parallel steps, one of two column shards", "M": M, "N_shard": half,
                          "storage": "bf16", "call": name, "us": round(ms * 1e3, 2), "bytes": nbytes,
                          "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), "max_diff_to_fwd": diff}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, help="a workload name, or 'all'")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=sorted(OP_CODES), default="softmax",
                    help="the row operation timed (softmax: the fused row softmax; rmsnorm, layernorm: the "
                         "normalisations on the same row engine)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-summary", action="store_true",
                    help="leave out the device-timed figures of the other workloads (all_configs) that the default "
                         "run adds to its line")
    ap.add_argument("--options", default=None,
                    help="JSON object of rs_options fields forcing a kernel configuration (tuning, profiling)")
    ap.add_argument("--rows", type=int, default=0,
                    help="use only the first ROWS rows of the workload (smaller profiler captures)")
    ap.add_argument("--causal", action="store_true",
                    help="softmax only: time rowsoftmax_causal_fwd with a square causal mask (row r keeps its first "
                         "(r mod N) + 1 elements, the rest is never read); bytes count the kept reads and all writes")
    ap.add_argument("--sweep-n", action="store_true",
                    help="instead of the benchmark line: the fp32 M=4096, N=256..12672 sweep of the row softmax, "
                         "one JSON line per (N, kernel configuration)")
    ap.add_argument("--sweep-wide", action="store_true",
                    help="instead of the benchmark line: 16-bit rows (N = 256..65536) of the --op row "
                         "operation through the planner's choice, the ring and the clusters (with --causal: the "
                         "causal softmax, mask period N)")
    ap.add_argument("--sweep-dtype", choices=["bf16", "f16"], default="bf16")
    ap.add_argument("--widths", default=None,
                    help="--sweep-wide: comma-separated row widths instead of 256..65536 (one width for a "
                         "profiler capture)")
    ap.add_argument("--split", action="store_true",
                    help="instead of the benchmark line: the split-row softmax (few wide rows through "
                         "rowsoftmax_split_fwd against rowsoftmax_fwd, and the vocabulary-parallel partial and "
                         "finish steps on two column shards of the bf16 causal scores)")
    args = ap.parse_args()
    args.options = json.loads(args.options) if args.options else None
    if args.causal and args.op != "softmax":
        raise SystemExit("--causal applies to the softmax only")
    if args.warmup < 3:
        args.warmup = 3
    args.summary_all = (args.workload == DEFAULT_WORKLOAD and not args.no_summary and not args.rows
                        and not args.options and not args.causal)
    from memory_bound_row_gb300 import workloads as W

    names = W.ORDER if args.workload == "all" else [args.workload]
    for n in names:
        if n not in W.WORKLOADS:
            raise SystemExit(f"unknown workload {n}; choose from {', '.join(W.ORDER)} or 'all'")
    if args.split:
        run_split(args)
    elif args.sweep_n:
        run_sweep_n(args)
    elif args.sweep_wide:
        run_sweep_wide(args)
    elif args.impl == "reference":
        run_reference(args, names)
    else:
        run_ours(args, names)


if __name__ == "__main__":
    main()
