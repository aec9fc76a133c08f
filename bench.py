"""Benchmark of the fused row softmax on GB300.

One step = one softmax_fwd call (the whole hot path: load, row max, exp and
sum, normalise and store, dispatch) over the largest workload of the pages
that fits one GPU: bf16 vocabulary logits, 512 x 131072 (Gumbel + Zipf(1.1)
offsets, seed 4; 268 MB moved per call).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c1..c5|wN] [--no-per-shape] [--no-sweep]

Timing: W warm-up steps, then exactly K steps bracketed by a barrier and a
device synchronisation.  The K launches are captured once into a CUDA graph;
the graph is replayed once untimed (its first replay uploads it) and then
once between CUDA events on the launching stream.  Each step reads a
different buffer set; the sets together are larger than 2.5x the L2, so every
step's input comes from HBM.  `value` is whole-job throughput (algorithmic
bytes 2*rows*cols*elem of all ranks / max-over-ranks time of the K steps);
the roofline block uses the same mean per-launch device time.  Under
torchrun every rank runs its own copy of the workload (weak scaling, rows
are independent: no data-path collective).

`per_shape` times every workload of the pages (and, unless --no-sweep, the
fp32 width sweep and the extra shapes of EXTRA_SHAPES) with the same graph
method: 200 launches after 50 warm-up.

The same line carries an `attention` object: the fused attention forward
(softmax_attention_fwd) on the pages' attention shapes (batch 4, 32 heads,
head dim 128, fp16, causal, N = 4096 and 16384) in TFLOP/s against the
measured dense tensor rate, with the oracle's one-head attention as its CPU
baseline.  `--attention KEY` prints only that object (with `--only-kernel`:
the command the attention profiler capture runs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 roofline (2×bytes/peak) per shape; µs/call"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED = 1900.0, 1700.0


# ---------------------------------------------------------------------------
# multi-rank plumbing (host side; tested on CPU with gloo)
# ---------------------------------------------------------------------------

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max_seconds(seconds: float, world: int) -> float:
    """Max of a per-rank duration over all ranks (identity when world == 1)."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_gbs(bytes_per_rank_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / max_seconds / 1e9


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t0 = self.t1 = 0.0

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except OSError:
            self.proc = None
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        self.t1 = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._reader.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None,
                "window_ms": round((self.t1 - self.t0) * 1e3, 1)}


def rotating_sets(x_dev, n_bytes_per_set: int, l2_bytes: int, min_sets: int = 2):
    """Buffer sets (in, out) totalling > 2.5x L2; the inputs are copies of x."""
    import torch
    sets = max(min_sets, -(-int(2.5 * l2_bytes) // max(1, n_bytes_per_set)))
    out = []
    for _ in range(sets):
        out.append((x_dev.clone(), torch.empty_like(x_dev)))
    return out


def time_steps(launch, sets, steps: int, warmup: int, world: int = 1, graph: bool = True):
    """W warm-up launches, then exactly `steps` launches over the rotating sets.

    With graph=True the timed launches are captured once into a CUDA graph and
    replayed, so the host's per-call cost (Python, ctypes, launch) cannot leave
    the GPU idle between steps.  The graph's first replay (which uploads it)
    runs untimed; events then bracket one replay on the launching stream.
    Returns (mean ms per launch, total ms, per-launch ms or None)."""
    import torch
    for i in range(warmup):
        launch(*sets[i % len(sets)])
    torch.cuda.synchronize()
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                launch(*sets[i % len(sets)])
        torch.cuda.synchronize()
        g.replay()  # upload: not part of the timed region
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    per = None
    if g is not None:
        t0.record()
        g.replay()
        t1.record()
    else:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        t0.record()
        for i in range(steps):
            starts[i].record()
            launch(*sets[i % len(sets)])
            ends[i].record()
        t1.record()
    torch.cuda.synchronize()
    barrier(world)
    total = t0.elapsed_time(t1)
    if g is None:
        per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    del g
    return total / steps, total, per


def traffic_record(workload: str):
    """ncu DRAM bytes per launch for this workload's dominant kernel, if the
    kernel sources are unchanged since the capture (else None)."""
    from memory_bound_row_softmax_gb300 import build as build_mod
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources_digest") != build_mod.sources_digest():
        return None
    return rec


L2_POLICY = "inputs larger than L2: each step reads another of a set of rotating buffers totalling > 2.5 x L2"


def workload_config(w, world: int) -> dict:
    """The `config` object of both arms' JSON lines (the same dict for the
    same workload and world size)."""
    return {"workload": w.name, "rows": w.rows, "cols": w.cols, "row_stride": w.stride,
            "storage_dtype": w.dtype, "parallelism": f"replicas x{world} (rows independent)", "l2": L2_POLICY}


def device_seeded(w, dev):
    """Input bits of w drawn on the device (timing-only workloads: the sweep
    and the extra shapes): U(lo, hi) or N(0, sigma^2) from torch's seeded
    device generator, rounded to the storage dtype."""
    import torch
    g = torch.Generator(device=dev).manual_seed(w.seed)
    if w.kind == "uniform":
        x = torch.rand((w.rows, w.stride), generator=g, device=dev) * (w.hi - w.lo) + w.lo
    else:
        x = torch.randn((w.rows, w.stride), generator=g, device=dev) * w.sigma
    if w.dtype == "f32":
        return x.view(torch.int32)
    return x.to(torch.float16 if w.dtype == "f16" else torch.bfloat16).view(torch.int16)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args) -> dict | None:
    import numpy as np
    import torch

    from memory_bound_row_softmax_gb300 import binding as B
    from memory_bound_row_softmax_gb300 import build as build_mod
    from memory_bound_row_softmax_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", init_method="env://")
    torch.cuda.set_device(local)
    build_mod.build()
    B.lib()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    peaks = measured_peaks()

    if args.attention:  # the attention forward alone (ncu captures, quick looks)
        if rank != 0:
            return None
        if args.only_kernel:
            w = W.ATTENTION_CONFIGS[args.attention]
            ms, _ = attention_time(w, dev, args.steps, args.warmup)
            print(json.dumps({"workload": w.name, "steps": args.steps, "ms_mean": ms,
                              "tflops": w.flops() / (ms / 1e3) / 1e12}))
            return None
        return {"attention": attention_block(peaks, dev, keys=(args.attention,))}

    if args.workload.startswith("w"):  # a width of the fp32 sweep, seeded on the device
        w = W.sweep_workload(int(args.workload[1:]))
        x = None
        x_dev = device_seeded(w, dev)
    elif args.workload in W.EXTRA_SHAPES:
        w = W.EXTRA_SHAPES[args.workload]
        x = None
        x_dev = device_seeded(w, dev)
    else:
        w = W.CONFIGS[args.workload]
        x = W.make_input(w)
        bits = x.view(np.int32 if w.dtype == "f32" else np.int16)
        x_dev = torch.from_numpy(bits).to(dev)
    code = B.DTYPE_CODES[w.dtype]
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    lib = B.lib()

    def launch(a, b):
        st = lib.softmax_fwd(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code,
                             torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise B.SoftmaxError(st)

    if args.masked:  # the workload's causal mask through softmax_fwd_masked (for --only-kernel captures)
        if not (args.only_kernel and w.causal_period):
            raise SystemExit("--masked needs --only-kernel and a causal workload (c4)")

        def launch(a, b):  # noqa: F811 -- the masked call replaces the plain one
            st = lib.softmax_fwd_masked(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code, 1.0, 0,
                                        w.causal_period, torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise B.SoftmaxError(st, "softmax_fwd_masked")

    if args.noalloc:  # the same rows through softmax_fwd_noalloc (for --only-kernel captures)
        if not args.only_kernel:
            raise SystemExit("--noalloc needs --only-kernel")

        def launch(a, b):  # noqa: F811 -- the allocation-free split replaces the plain call
            st = lib.softmax_fwd_noalloc(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code,
                                         torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise B.SoftmaxError(st, "softmax_fwd_noalloc")

    if args.force:
        B.set_force_path(*[int(v) for v in args.force.split(",")])
    B.set_launch_overlap(not args.no_overlap)
    plan = B.plan(x_dev.data_ptr(), x_dev.data_ptr() + (1 << 40), w.rows, w.cols, w.stride, code)
    set_bytes = 2 * x_dev.numel() * x_dev.element_size()
    sets = rotating_sets(x_dev, set_bytes, l2)

    if args.only_kernel:  # the command the ncu captures run: eager launches only
        mean_ms, total_ms, _ = time_steps(launch, sets, args.steps, args.warmup, world, graph=False)
        if rank == 0:
            print(json.dumps({"workload": w.name, "steps": args.steps, "us_mean": mean_ms * 1e3, "plan": plan}))
        return None

    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local)
    clocks.start()
    # untimed pre-load so that the clock samples see this kernel's steady state
    t_end = time.time() + 0.4
    while time.time() < t_end:
        for i in range(200):
            launch(*sets[i % len(sets)])
        torch.cuda.synchronize()
    mean_launch_ms, total_ms, _ = time_steps(launch, sets, args.steps, args.warmup, world)
    clk = clocks.stop()

    max_s = reduce_max_seconds(total_ms / 1e3, world)
    alg = w.algorithmic_bytes
    value = aggregate_gbs(alg, args.steps, world, max_s)
    achieved = plan["hbm_bytes"] / (mean_launch_ms / 1e3) / 1e9
    traffic = traffic_record(w.name)
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(w, world),
        "timing": {
            "method": "K launches captured in one CUDA graph; one untimed replay (graph upload), then one "
                      "replay between CUDA events on the launching stream",
            "buffer_sets": len(sets), "buffer_bytes": len(sets) * set_bytes, "l2_bytes": l2,
            "launch_overlap": not args.no_overlap, "arithmetic": "f32 (one exp per element)",
        },
        "plan": {"path": B.PATH_NAMES.get(plan["path"]), "threads": plan["threads"], "vpt": plan["vpt"],
                 "group": plan["group"], "grid": plan["grid"]},
        "us_per_call": round(mean_launch_ms * 1e3, 3),
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
            "traffic": traffic["bytes_per_launch"] if traffic else None,
            "algorithmic_bytes": plan["hbm_bytes"],
        },
        "clocks": clk,
        "gpu_launches": args.steps * plan["launches"],
    }
    if rank == 0 and x is not None:
        result["e2e"] = e2e_measure(x, w, dev, min(args.steps, 2000))
    if rank == 0 and world == 1 and not args.no_cpu_baseline and x is not None:
        result["cpu_baseline"] = cpu_baseline(x, w)
    if rank == 0 and world == 1 and not args.no_per_shape:
        result["per_shape"] = per_shape(args, peaks, l2, dev)
    if rank == 0 and world == 1 and not args.no_attention:
        result["attention"] = attention_block(peaks, dev)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


def e2e_measure(x, w, dev, steps: int) -> dict:
    """Same metric through the C ABI with host buffers: softmax_fwd_host on a
    page-locked input and output every step, all inside the timed region.
    The headline value is its zero-copy mode (the kernels read the input and
    write the output across the CPU-GPU link themselves); `staged` is its
    device-workspace mode (host-to-device copies, the softmax and the
    device-to-host copies, chunked and overlapped by the library).  Beside
    them, the link ceiling: the same bytes copied host-to-device and
    device-to-host at once (two streams, one copy each way per step, no
    kernel), timed the same way."""
    import numpy as np
    import torch

    from memory_bound_row_softmax_gb300 import binding as B
    bits = x.view(np.int32 if w.dtype == "f32" else np.int16)
    h_in = torch.from_numpy(bits).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    code = B.DTYPE_CODES[w.dtype]
    ws = torch.empty(B.host_workspace_bytes(w.rows, w.cols, w.stride, code), dtype=torch.uint8, device=dev)
    lib = B.lib()
    stream = torch.cuda.current_stream(dev).cuda_stream

    def step():  # zero-copy: the kernels read and write the page-locked buffers in place
        st = lib.softmax_fwd_host(h_in.data_ptr(), h_out.data_ptr(), w.rows, w.cols, w.stride, code, None, 0,
                                  stream)
        if st != 0:
            raise B.SoftmaxError(st, "softmax_fwd_host")

    def step_staged():  # the three-slot copy / softmax / copy pipeline through a device workspace
        st = lib.softmax_fwd_host(h_in.data_ptr(), h_out.data_ptr(), w.rows, w.cols, w.stride, code, ws.data_ptr(),
                                  ws.numel(), stream)
        if st != 0:
            raise B.SoftmaxError(st, "softmax_fwd_host")

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(n):
            fn()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    ms = timed(step, steps)
    ms_staged = timed(step_staged, steps)
    # the link ceiling: H2D of the input and D2H of an output-sized buffer,
    # concurrently on two streams, both ordered after the current stream
    d_a, d_b = torch.empty_like(h_in, device=dev), torch.empty_like(h_in, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cur = torch.cuda.current_stream(dev)

    def duplex():
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s_out):
            h_out.copy_(d_b, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    dms = timed(duplex, steps)
    nbytes = h_in.numel() * h_in.element_size()
    value = w.algorithmic_bytes / (ms / 1e3) / 1e9
    ceiling = w.algorithmic_bytes / (dms / 1e3) / 1e9
    del d_a, d_b, ws
    return {"value": round(value, 2), "unit": "GB/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "steps": steps,
            "ms_per_step": round(ms, 4),
            "call": "softmax_fwd_host, zero-copy mode (no workspace): the kernels read the page-locked input and "
                    "write the page-locked output over the CPU-GPU link, each byte crossing it once",
            "staged": {"value": round(w.algorithmic_bytes / (ms_staged / 1e3) / 1e9, 2), "unit": "GB/s",
                       "ms_per_step": round(ms_staged, 4),
                       "call": "softmax_fwd_host with its recommended device workspace (copy / softmax / copy "
                               "pipeline over three slots)"},
            "link_ceiling": {"value": round(ceiling, 2), "unit": "GB/s", "ms_per_step": round(dms, 4),
                             "what": "the same bytes copied host-to-device and device-to-host at once "
                                     "(pinned memory, two streams, no kernel)"},
            "frac_of_link": round(value / ceiling, 4)}


def cpu_baseline(x, w, seconds: float = 4.0) -> dict:
    """The CPU oracle (untuned) on the workload: once on one thread over a
    bounded sample of its rows, once row-partitioned over every host core the
    process can use (whole passes over all rows, at least `seconds`)."""
    import oracle
    cores = os.cpu_count() or 1
    # one thread: rows [0, n) with n sized to about `seconds`
    n = max(1, min(w.rows, 8))
    t0 = time.perf_counter()
    oracle.softmax(x[:n], w.dtype, cols=w.cols, threads=1)
    per_row = (time.perf_counter() - t0) / n
    n1 = int(max(1, min(w.rows, seconds / max(per_row, 1e-9))))
    t0 = time.perf_counter()
    oracle.softmax(x[:n1], w.dtype, cols=w.cols, threads=1)
    el1 = time.perf_counter() - t0
    one = {"value": round(2 * n1 * w.cols * w.elem_bytes / el1 / 1e9, 4), "unit": "GB/s", "cores": 1,
           "elements_per_s": round(n1 * w.cols / el1), "wall_ms": round(el1 * 1e3, 1),
           "sample": f"rows 0..{n1 - 1} of {w.name} ({n1} of {w.rows} rows, {el1:.1f} s)"}
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.softmax(x, w.dtype, cols=w.cols, threads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": round(w.algorithmic_bytes * reps / el / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "elements_per_s": round(reps * w.rows * w.cols / el),
            "wall_ms_per_pass": round(el / reps * 1e3, 1),
            "sample": f"{reps} full pass(es) over all {w.rows} rows of {w.name} ({el:.1f} s wall, "
                      f"double-precision C, rows split over {cores} threads = os.cpu_count() of this "
                      f"process, which may be a container's share of the host)",
            "single_thread": one}


def per_shape(args, peaks, l2, dev) -> dict:
    """Every workload of the pages (and, unless --no-sweep, the fp32 width
    sweep and the extra shapes): mean us/call over 200 timed launches after 50
    warm-up (the harness of the pages; replayed from a CUDA graph), GB/s,
    fraction of the measured HBM peak and of a device-to-device copy of the
    same bytes timed the same way.  The few-long-row shapes also time
    softmax_fwd_noalloc (the grid-wide split path)."""
    import numpy as np
    import torch

    from memory_bound_row_softmax_gb300 import binding as B
    from memory_bound_row_softmax_gb300 import workloads as W

    lib = B.lib()
    todo = [W.CONFIGS[k] for k in ("c1", "c2", "c3", "c4", "c5")]
    if not args.no_sweep:
        todo += list(W.EXTRA_SHAPES.values()) + [W.sweep_workload(c) for c in W.SWEEP_WIDTHS]
    table = {}
    for w in todo:
        if w.name.startswith("c"):
            x = W.make_input(w)
            xd = torch.from_numpy(x.view(np.int32 if w.dtype == "f32" else np.int16)).to(dev)
        else:  # timing-only matrices: seeded on the device
            xd = device_seeded(w, dev)
        code = B.DTYPE_CODES[w.dtype]

        def launch(a, b, w=w, code=code):
            st = lib.softmax_fwd(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code,
                                 torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise B.SoftmaxError(st)

        plan = B.plan(xd.data_ptr(), xd.data_ptr() + (1 << 40), w.rows, w.cols, w.stride, code)
        set_bytes = 2 * xd.numel() * xd.element_size()
        sets = rotating_sets(xd, set_bytes, l2)
        med, _, _ = time_steps(launch, sets, 200, 50)
        # the same launches in plain stream order (no launch overlap)
        B.set_launch_overlap(False)
        med_plain, _, _ = time_steps(launch, sets, 200, 50)
        B.set_launch_overlap(not args.no_overlap)
        # after softmax_autotune on this shape (its cache entry is dropped again)
        tuned = B.autotune_ptr(sets[0][0].data_ptr(), sets[0][1].data_ptr(), w.rows, w.cols, w.stride, code,
                               torch.cuda.current_stream().cuda_stream, iters=20)
        med_tuned, _, _ = time_steps(launch, sets, 200, 50)
        B.autotune_clear()
        # the copy ceiling: rows*cols*elem bytes, device to device, same
        # rotation; the size is rounded down to 64 KiB because the runtime's
        # copy runs at half speed on sizes that are not (200,000,000 bytes:
        # 131 us, 199,950,336 bytes: 60 us)
        nbytes = max(65536, (w.rows * w.cols * w.elem_bytes) // 65536 * 65536)
        nwords = nbytes // 4
        csets = [(torch.empty(nwords, dtype=torch.int32, device=dev), torch.empty(nwords, dtype=torch.int32, device=dev))
                 for _ in range(max(2, -(-int(2.5 * l2) // (8 * nwords))))]
        cmed, _, _ = time_steps(lambda a, b: b.copy_(a), csets, 200, 50)
        gbs = plan["hbm_bytes"] / (med / 1e3) / 1e9
        alg = w.algorithmic_bytes / (med / 1e3) / 1e9
        copy_gbs = 2 * nbytes / (cmed / 1e3) / 1e9
        row = {
            "path": B.PATH_NAMES.get(plan["path"]),
            "shape": [plan["threads"], plan["vpt"], plan["group"]],
            "us_per_call": round(med * 1e3, 2),
            "us_per_call_no_overlap": round(med_plain * 1e3, 2),
            "us_per_call_tuned": round(med_tuned * 1e3, 2),
            "tuned_shape": [tuned["plan"][k] for k in ("path", "threads", "vpt", "group")],
            "gbs": round(alg, 1), "frac_of_measured_hbm": round(alg / peaks["hbm_gbs"], 4),
            "frac_of_nominal_8tbs": round(alg / 8000.0, 4),
            "copy_us": round(cmed * 1e3, 2), "copy_gbs": round(copy_gbs, 1),
            "frac_of_copy": round(alg / copy_gbs, 4), "time_vs_copy": round(med / cmed, 3),
            "moved_gbs": round(gbs, 1),
        }
        if w.rows * 16 < 152:  # a few very long rows: the grid-wide split through softmax_fwd_noalloc
            def launch_noalloc(a, b, w=w, code=code):
                st = lib.softmax_fwd_noalloc(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code,
                                             torch.cuda.current_stream().cuda_stream)
                if st != 0:
                    raise B.SoftmaxError(st, "softmax_fwd_noalloc")

            nmed, _, _ = time_steps(launch_noalloc, sets, 200, 50)
            row["us_per_call_noalloc_split"] = round(nmed * 1e3, 2)
        table[w.name] = row
        if w.causal_period:  # the same rows through softmax_fwd_masked: only the kept half is read
            def launch_masked(a, b, w=w, code=code):
                st = lib.softmax_fwd_masked(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code, 1.0, 0,
                                            w.causal_period, torch.cuda.current_stream().cuda_stream)
                if st != 0:
                    raise B.SoftmaxError(st, "softmax_fwd_masked")

            mmed, _, _ = time_steps(launch_masked, sets, 200, 50)
            masked_path = B.last_path()
            kept = sum(min(w.cols, (r % w.causal_period) + 1) for r in range(w.rows))
            mbytes = (kept + w.rows * w.cols) * w.elem_bytes  # kept entries read, every entry written
            entry = {
                "path": "masked " + B.PATH_NAMES.get(masked_path, "?"), "us_per_call": round(mmed * 1e3, 2),
                "algorithmic_bytes": mbytes, "gbs": round(mbytes / (mmed / 1e3) / 1e9, 1),
                "frac_of_measured_hbm": round(mbytes / (mmed / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                "time_vs_unmasked": round(mmed / med, 3),
            }
            if masked_path == B.PATH_CTA:
                # the same access pattern with no arithmetic, one block of the
                # masked call's size per row: kept entries copied, the rest zeroed
                pthreads = B.plan(sets[0][0].data_ptr(), sets[0][1].data_ptr(), w.rows, w.cols, w.stride,
                                  w.dtype)["threads"]

                def launch_pattern(a, b, w=w, code=code, pthreads=pthreads):
                    st = B.masked_copy_ptr(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code, 0,
                                           w.causal_period, pthreads, torch.cuda.current_stream().cuda_stream)
                    if st != 0:
                        raise B.SoftmaxError(st, "softmax_masked_copy")

                pmed, _, _ = time_steps(launch_pattern, sets, 200, 50)
                entry["pattern_copy_us"] = round(pmed * 1e3, 2)
                entry["time_vs_pattern_copy"] = round(mmed / pmed, 3)

                # the writes alone: the same kernel with nothing kept (every
                # output written as zero, no input read)
                def launch_writes(a, b, w=w, code=code, pthreads=pthreads):
                    st = B.masked_copy_ptr(a.data_ptr(), b.data_ptr(), w.rows, w.cols, w.stride, code,
                                           -(w.cols + 1), w.causal_period, pthreads,
                                           torch.cuda.current_stream().cuda_stream)
                    if st != 0:
                        raise B.SoftmaxError(st, "softmax_masked_copy")

                zmed, _, _ = time_steps(launch_writes, sets, 200, 50)
                entry["writes_only_us"] = round(zmed * 1e3, 2)
            table[w.name + "_masked"] = entry
        del sets, csets, xd
        torch.cuda.empty_cache()
    return table


# ---------------------------------------------------------------------------
# the fused attention forward (softmax_attention_fwd)
# ---------------------------------------------------------------------------

def attention_inputs(w, dev):
    """Q, K, V ~ N(0, 1) from a seeded device generator, rounded to the dtype."""
    import torch
    g = torch.Generator(device=dev).manual_seed(w.seed)
    shape = (w.batch, w.heads, w.n_ctx, w.head_dim)
    tdt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    return tuple(torch.randn(shape, generator=g, device=dev).to(tdt) for _ in range(3))


def attention_time(w, dev, steps: int, warmup: int) -> tuple[float, int]:
    """Mean ms per softmax_attention_fwd call over `steps` eager launches
    bracketed by CUDA events on the launching stream (Q, K and V together are
    larger than L2 for the benchmarked sizes)."""
    import torch

    from memory_bound_row_softmax_gb300 import binding as B
    q, k, v = attention_inputs(w, dev)
    o = torch.empty_like(q)
    lib = B.lib()
    code = B.DTYPE_CODES[w.dtype]
    scale = 1.0 / w.head_dim ** 0.5

    def launch():
        st = lib.softmax_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), w.batch, w.heads,
                                       w.n_ctx, w.head_dim, code, 1 if w.causal else 0, scale,
                                       torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise B.SoftmaxError(st, "softmax_attention_fwd")

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        launch()
    t1.record()
    torch.cuda.synchronize()
    if B.check_device_error() != B.OK:
        raise RuntimeError("attention kernel reported a device error")
    nbytes = 4 * q.numel() * q.element_size()
    del q, k, v, o
    torch.cuda.empty_cache()
    return t0.elapsed_time(t1) / steps, nbytes


def attention_cpu_baseline(w, rows: int = 48) -> dict:
    """The oracle's one-head attention (double precision, one thread) on the
    last `rows` queries of one head of the workload (the rows with the most
    keys under the causal mask), in matmul FLOPs per second."""
    import oracle
    from memory_bound_row_softmax_gb300 import workloads as W
    q = W.qkv_heads(w.seed, "q", 0, 1, w.n_ctx, w.head_dim, w.dtype)[0]
    k = W.qkv_heads(w.seed, "k", 0, 1, w.n_ctx, w.head_dim, w.dtype)[0]
    v = W.qkv_heads(w.seed, "v", 0, 1, w.n_ctx, w.head_dim, w.dtype)[0]
    r0 = w.n_ctx - rows
    t0 = time.perf_counter()
    oracle.attention_fwd(q[r0:], k, v, w.dtype, 1.0 / w.head_dim ** 0.5, causal=w.causal, causal_offset=r0)
    el = time.perf_counter() - t0
    keys = sum(min(w.n_ctx, r + 1) if w.causal else w.n_ctx for r in range(r0, w.n_ctx))
    flops = 4.0 * keys * w.head_dim
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"queries {r0}..{w.n_ctx - 1} of head 0 of {w.name} ({keys} query-key pairs, "
                      f"{el:.2f} s, double-precision C, one thread)"}


def attention_block(peaks, dev, keys=("a4k", "a16k")) -> dict:
    """Per workload: ms per call, TFLOP/s (4 B H N^2 D, halved when causal) and
    the tensor roofline (the measured bf16 dense GEMM rate; fp16 runs at the
    same nominal rate)."""
    from memory_bound_row_softmax_gb300 import workloads as W
    out = {"call": "softmax_attention_fwd", "workloads": {}}
    for key in keys:
        w = W.ATTENTION_CONFIGS[key]
        ms, nbytes = attention_time(w, dev, steps=20 if w.n_ctx <= 4096 else 10, warmup=3)
        tf = w.flops() / (ms / 1e3) / 1e12
        out["workloads"][w.name] = {
            "batch": w.batch, "heads": w.heads, "n_ctx": w.n_ctx, "head_dim": w.head_dim, "dtype": w.dtype,
            "causal": w.causal, "ms_per_call": round(ms, 4), "tflops": round(tf, 1),
            "flops_per_call": w.flops(), "hbm_bytes_min": nbytes,
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops_sustained"],
                         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops_sustained"], 4),
                         "peak_kind": "sustained (back-to-back launches)",
                         "frac_of_burst": round(tf / peaks["bf16_tflops"], 4), "peak_source": peaks["source"]},
        }
    out["cpu_baseline"] = attention_cpu_baseline(W.ATTENTION_CONFIGS[keys[0]])
    return out


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle, as it stands
# ---------------------------------------------------------------------------

def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    from memory_bound_row_softmax_gb300 import workloads as W
    oracle.build()
    if args.workload.startswith("w"):
        w = W.sweep_workload(int(args.workload[1:]))
    else:
        w = W.EXTRA_SHAPES[args.workload] if args.workload in W.EXTRA_SHAPES else W.CONFIGS[args.workload]
    x = W.make_input(w)
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.softmax(x, w.dtype, cols=w.cols, threads=cores)
    t_full = time.perf_counter() - t0
    budget_s = 90.0
    rows_per_step = int(max(1, min(w.rows, w.rows * budget_s / max(1, args.steps + args.warmup) / t_full)))
    for i in range(args.warmup):
        r0 = (i * rows_per_step) % max(1, w.rows - rows_per_step + 1)
        oracle.softmax(x[r0:r0 + rows_per_step], w.dtype, cols=w.cols, threads=cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        r0 = (i * rows_per_step) % max(1, w.rows - rows_per_step + 1)
        oracle.softmax(x[r0:r0 + rows_per_step], w.dtype, cols=w.cols, threads=cores)
    el = time.perf_counter() - t0
    step_bytes = 2 * rows_per_step * w.cols * w.elem_bytes
    value = step_bytes * args.steps / el / 1e9
    sample = (f"each step: rows [r0, r0+{rows_per_step}) of {w.name} ({rows_per_step} of {w.rows} rows), "
              f"double-precision C oracle over {cores} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="c5",
                    help="c1..c5 (the pages' workloads), r1, r2, l1..l3 (the extra shapes) or wN (fp32 "
                         "width-sweep matrix of width N)")
    ap.add_argument("--no-per-shape", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave the fp32 width sweep and the extra shapes out of the per-shape table")
    ap.add_argument("--force", default="",
                    help="path[,threads,vpt,group]: force a kernel path and launch shape (profiling, tuning)")
    ap.add_argument("--masked", action="store_true",
                    help="with --only-kernel on c4: run its causal mask through softmax_fwd_masked")
    ap.add_argument("--noalloc", action="store_true",
                    help="with --only-kernel: run the workload through softmax_fwd_noalloc (the split path)")
    ap.add_argument("--only-kernel", action="store_true",
                    help="warm-up and timed launches only (the command profiled with ncu)")
    ap.add_argument("--no-attention", action="store_true", help="leave out the attention forward block")
    ap.add_argument("--attention", default="",
                    help="a4k | a16k | a4k_small | a4k_wave: time only the fused attention forward on that workload")
    ap.add_argument("--json-out", default="")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch in plain stream order (no programmatic dependent launch)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        line = json.dumps(res)
        print(line, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(line + "\n")


if __name__ == "__main__":
    main()
