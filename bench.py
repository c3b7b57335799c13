"""Benchmark of the fused GEMM + epilogue on one GB300 (or N replicas, one per GPU).

A step is one call of the fused kernel over one batch of synthetic input: by default the
4096 x 4096 x 4096 bf16 GEMM + bias + ReLU.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
  python bench.py --sweep          # every workload (+ unfused chain, GROUP sweep) -> stderr + JSON

Timing: inputs rotate over several independent sets whose total exceeds twice the L2 size, so
every step reads A and B from HBM; CUDA events on the launching stream; barrier + synchronize on
both sides of the timed region; the maximum over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused GEMM+epilogue TFLOP/s and % of dense BF16 tensor peak (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES_DEFAULT = 129 * 1024 * 1024


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


SUSTAINED_S = 0.5  # a timed region at least this long is held against the sustained peak


def tensor_peak(pk, w, sustained=False):
    """Dense tensor peak for the workload's operand type: the measured bf16 figure (the burst one
    for a kernel timed briefly, the sustained one, taken back to back for seconds under the power
    cap, for a timed region of SUSTAINED_S or more), times the nominal fp8 / bf16 ratio
    (4.5 / 2.25) for fp8 operands."""
    from gemm_epilogue_gb300 import inputs as gen
    key = "bf16_tflops_sustained" if sustained and "bf16_tflops_sustained" in pk else "bf16_tflops"
    return pk[key] * (2.0 if w.ab_type == gen.E4M3 else 1.0)


def strip_comments(src: str) -> str:
    """C / C++ source without its comments (string literals kept), so that the hash below follows
    the code only."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


# The sources a kernel's DRAM traffic depends on: its own file, the shared device helpers and
# parameter structs, and the host code that plans and launches it.
KERNEL_SOURCES = {
    "tc_gemm_kernel": ["api.cu", "kernels.h", "ptx.cuh", "tc_gemm.cu", "tile_order.h"],
    "skinny_kernel": ["api.cu", "kernels.h", "ptx.cuh", "skinny.cu"],
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of a kernel's device and launch code (every source file when `kernel` is None;
    comments and layout excluded): recorded ncu traffic counts only while this matches the hash
    stored with it."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gemm_epilogue_gb300", "csrc")
    files = KERNEL_SOURCES[kernel] if kernel else sorted(os.listdir(d))
    for f in files:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            code = " ".join(strip_comments(fh.read()).split())  # layout and comments excluded
            h.update(f.encode() + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs.  Each sample
    carries nvidia-smi's own timestamp (local wall clock), so that only the samples taken inside
    the timed window count."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.rows = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    @staticmethod
    def _when(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, window=None):
        """Summary of the samples taken inside `window` = (t0, t1) in time.time() seconds (all
        samples when None)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                self.rows.append({"t": self._when(parts[0]), "sm": float(parts[2]),
                                  "max": float(parts[3]),
                                  "power": float(parts[4]) if parts[4] not in ("[N/A]", "") else 0.0,
                                  "hw_slow": parts[6], "hw_therm": parts[7], "sw_therm": parts[8],
                                  "sw_power": parts[9]})
            except ValueError:
                continue
        rows = self.rows
        if window is not None:
            t0, t1 = window
            rows = [r for r in rows if r["t"] is not None and t0 <= r["t"] <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_total": len(self.rows)}
        reasons = set()
        for r in rows:
            for k, name in (("hw_slow", "hw_slowdown"), ("hw_therm", "hw_thermal_slowdown"),
                            ("sw_therm", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[k] == "Active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_total": len(self.rows),
                "power_w_median": statistics.median(r["power"] for r in rows),
                "window": "samples taken inside the timed replays"}


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def slowest_rank(dist, value, device=None):
    """Max over the ranks of a per-rank time: every rank times its own replica of the workload,
    and the job takes as long as its slowest rank.  `dist` is torch.distributed (None: one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- our implementation

class Problem:
    """Device-resident rotating input sets of one workload, and a call of the fused kernel."""

    def __init__(self, w, dev, l2_bytes, max_sets=8, with_unfused=False):
        import torch
        from gemm_epilogue_gb300 import inputs as gen
        import gemm_epilogue_gb300.binding as fg
        self.w, self.dev, self.fg = w, dev, fg
        tdt = {gen.F16: torch.float16, gen.BF16: torch.bfloat16, gen.F32: torch.float32,
               gen.E4M3: torch.uint8}
        self.tdt = tdt
        x = gen.make(w)
        self.host = x

        def up(a, t):
            if a is None:
                return None
            if t in (gen.F32, gen.E4M3):
                return torch.from_numpy(a).to(dev)
            return torch.from_numpy(a.view(np.int16)).view(tdt[t]).to(dev)

        A, B = up(x.A, w.ab_type), up(x.B, w.ab_type)
        bias, Y = up(x.bias, w.bias_type), up(x.Y, w.y_type)
        set_bytes = A.numel() * A.element_size() + B.numel() * B.element_size()
        set_bytes += w.M * w.N * gen.ELEM_BYTES[w.out_type] * (2 if Y is not None else 1)
        n = max(1, min(max_sets, math.ceil(2 * l2_bytes / max(set_bytes, 1)) + 1))
        self.sets = []
        for i in range(n):
            if i == 0:
                a, b, y = A, B, Y
            else:  # independent copies (same values, different addresses)
                a, b = A.clone(), B.clone()
                y = Y.clone() if Y is not None else None
            out = torch.empty(w.M, w.N, dtype=tdt[w.out_type], device=dev)
            self.sets.append((a, b, bias, y, out))
        self.set_bytes = set_bytes
        self.word = {gen.F16: fg.F16, gen.BF16: fg.BF16, gen.E4M3: fg.E4M3}[w.ab_type]
        if w.bias_type == gen.F32:
            self.word |= fg.BIAS_F32
        elif w.bias_type == gen.BF16 and w.ab_type != gen.BF16:
            self.word |= fg.BIAS_BF16
        if w.out_type == gen.F32:
            self.word |= fg.OUT_F32
        elif w.out_type == gen.BF16 and w.ab_type != gen.BF16:
            self.word |= fg.OUT_BF16
        elif w.out_type == gen.F16 and w.ab_type != gen.F16:
            self.word |= fg.OUT_F16
        if w.epilogue == "gate" and w.y_type != w.ab_type:
            self.word |= {gen.F16: fg.Y_F16, gen.BF16: fg.Y_BF16}[w.y_type]
        self.ws = None
        if with_unfused:
            nb = fg.fgemm_unfused_workspace_bytes(w.M, w.N, self.word, 0)
            self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            self.ws_bytes = nb

    def plan(self, opts=None):
        a, b, bias, y, out = self.sets[0]
        w = self.w
        return self.fg.fgemm_plan(a, b, bias, y, out, w.M, w.N, w.K, self.word,
                                  gate=y is not None, opts=opts)

    def call(self, i, stream, opts=None, unfused=False):
        a, b, bias, y, out = self.sets[i % len(self.sets)]
        w, fg = self.w, self.fg
        if unfused:
            if y is not None:
                fg.fgemm_unfused_addmm_gate(a, b, bias, y, out, w.M, w.N, w.K, self.word, self.ws,
                                            self.ws_bytes, 0, stream)
            else:
                fg.fgemm_unfused_bias_relu(a, b, bias, out, w.M, w.N, w.K, self.word, self.ws,
                                           self.ws_bytes, 0, stream)
            return None
        if y is not None:
            return fg.fgemm_addmm_gate_ex(a, b, bias, y, out, w.M, w.N, w.K, self.word, stream, opts)
        return fg.fgemm_bias_relu_ex(a, b, bias, out, w.M, w.N, w.K, self.word, stream, opts)


def time_steps(prob, steps, warmup, stream, opts=None, unfused=False, barrier=None):
    import torch
    path = None
    for i in range(warmup):
        path = prob.call(i, stream.cuda_stream, opts, unfused)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        path = prob.call(warmup + i, stream.cuda_stream, opts, unfused)
    end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(end) / steps, path


def time_steps_graph(prob, steps, warmup, stream, barrier=None, opts=None, min_seconds=1.0):
    """The timed steps of the bench line: `warmup` untimed calls on the stream, then the next
    `steps` calls (the same rotation of input sets as the stream loop) captured once in a CUDA
    graph, so that the host's and the driver's per-launch gaps do not sit between the steps.
    The graph is replayed back to back, each replay between its own pair of CUDA events on the
    launching stream, until the replays have kept the GPU busy for `min_seconds` (at least 5
    replays); the time per step is the median replay time / `steps`.  Every step runs in full.
    Returns (ms per step, path, replays, (t0, t1) wall-clock window of the replays)."""
    import torch
    path = None
    for i in range(warmup):
        path = prob.call(i, stream.cuda_stream, opts)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    # thread_local: CUDA calls of other threads (NCCL's watchdog under torchrun) do not void it
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(steps):
            path = prob.call(warmup + i, stream.cuda_stream, opts)
    torch.cuda.synchronize()
    # one timed replay to size the run
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    one = max(e0.elapsed_time(e1) * 1e-3, 1e-6)
    reps = max(5, min(20000, int(math.ceil(min_seconds / one))))
    if barrier:
        barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    t0 = time.time()
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if barrier:
        barrier()
    per = sorted(a.elapsed_time(b) for a, b in ev)
    return statistics.median(per) / steps, path, reps, (t0, t1)


def time_graph(prob, steps, warmup, stream, opts=None, reps=5):
    """Device time per call with host launch overhead removed: `steps` calls captured once in a
    CUDA graph, the graph replayed `reps` times between CUDA events."""
    import torch
    for i in range(warmup):
        prob.call(i, stream.cuda_stream, opts)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(steps):
            prob.call(i, stream.cuda_stream, opts)
    g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / (steps * reps)


def e2e_steps(prob, steps, stream):
    """End to end through the C ABI: each step uploads its own A, B, bias (and Y) from pinned host
    memory, runs the fused call and reads its output back into pinned host memory.  Consecutive
    steps are pipelined the way a serving loop would run them: two device buffer sets alternate,
    the upload of step i + 1 (A and B on two copy streams) overlaps the call and the read-back of
    step i, and events keep every buffer's reuse in order.  The timed region spans all copies.
    (Four upload streams measured no faster: host-to-device runs at about 190 GB/s either way.)"""
    import torch
    w = prob.w
    sets = prob.sets[:2]
    fg = prob.fg
    a0, b0, bias0, y0, _ = sets[0]
    hA = torch.empty_like(a0, device="cpu").pin_memory()
    hB = torch.empty_like(b0, device="cpu").pin_memory()
    hb = torch.empty_like(bias0, device="cpu").pin_memory()
    hY = torch.empty_like(y0, device="cpu").pin_memory() if y0 is not None else None
    hA.copy_(a0)
    hB.copy_(b0)
    hb.copy_(bias0)
    if hY is not None:
        hY.copy_(y0)
    host_out = [torch.empty_like(s_[4], device="cpu").pin_memory() for s_ in sets]
    h2d = sum(t.numel() * t.element_size() for t in (hA, hB, hb, hY) if t is not None)
    d2h = host_out[0].numel() * host_out[0].element_size()
    dev = a0.device
    up_a = torch.cuda.Stream(device=dev)
    up_b = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    ev = torch.cuda.Event
    computed = [ev() for _ in sets]      # call on set j finished (its inputs free again)
    read_back = [ev() for _ in sets]     # output of set j copied to the host (out free again)
    for e_ in computed + read_back:
        e_.record(stream)

    def one(i):
        j = i % 2
        a, b, bias, y, out = sets[j]
        up_a.wait_event(computed[j])
        up_b.wait_event(computed[j])
        with torch.cuda.stream(up_a):
            a.copy_(hA, non_blocking=True)
            bias.copy_(hb, non_blocking=True)
        with torch.cuda.stream(up_b):
            b.copy_(hB, non_blocking=True)
            if hY is not None:
                y.copy_(hY, non_blocking=True)
        e_a, e_b = ev(), ev()
        e_a.record(up_a)
        e_b.record(up_b)
        stream.wait_event(e_a)
        stream.wait_event(e_b)
        stream.wait_event(read_back[j])
        if y is not None:
            fg.fgemm_addmm_gate(a, b, bias, y, out, w.M, w.N, w.K, prob.word, stream.cuda_stream)
        else:
            fg.fgemm_bias_relu(a, b, bias, out, w.M, w.N, w.K, prob.word, stream.cuda_stream)
        computed[j].record(stream)
        down.wait_event(computed[j])
        with torch.cuda.stream(down):
            host_out[j].copy_(out, non_blocking=True)
        read_back[j].record(down)

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(up_a)
    for u in (up_b, stream, down):
        u.wait_event(start)
    for i in range(steps):
        one(i)
    for e_ in read_back:
        up_a.wait_event(e_)
    end.record(up_a)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


def cpu_baseline(w, target_s=12.0):
    """The fp64 oracle as it stands, on a bounded row sample of the same workload."""
    import oracle
    from gemm_epilogue_gb300 import inputs as gen
    oracle.build()
    x = gen.make(w)
    threads = oracle.default_threads()
    rows = max(1, min(w.M, threads))
    while True:
        sel = np.arange(rows, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.gemm_epilogue(x.A, x.B, x.bias, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type,
                             oracle.EPI_GATE if w.epilogue == "gate" else oracle.EPI_RELU,
                             Y=x.Y, rows=sel, threads=threads, want_ref=False, y_type=w.y_type)
        dt = time.perf_counter() - t0
        if dt >= target_s / 4 or rows >= w.M:
            break
        rows = min(w.M, max(rows + 1, int(rows * min(8.0, target_s / max(dt, 1e-3)))))
    tflops = 2.0 * rows * w.N * w.K / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {w.M} output rows of {w.name} (all {w.N} columns, K={w.K}), "
                      f"{dt:.2f} s", "seconds": dt}


def run_ours(args):
    import torch
    from gemm_epilogue_gb300 import build as libbuild
    from gemm_epilogue_gb300 import inputs as gen
    rank, world, local = env_rank()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        libbuild.build()
    if dist:
        dist.barrier()
    import gemm_epilogue_gb300.binding as fg
    fg.lib()
    w = gen.WORKLOADS[args.workload]
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_DEFAULT
    prob = Problem(w, dev, l2, with_unfused=args.variant == "unfused")
    stream = torch.cuda.Stream(device=dev)
    barrier = (lambda: dist.barrier()) if dist else None
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    unfused = args.variant == "unfused"
    opts = json.loads(args.opts) if args.opts else None
    window = None
    reps = 1
    if unfused:  # the library's comparison chain: launched from the stream loop
        t0 = time.time()
        ms, path = time_steps(prob, args.steps, args.warmup, stream, barrier=barrier, unfused=True)
        window = (t0, time.time())
        ms_loop = ms
        launch = "stream loop"
    else:
        ms, path, reps, window = time_steps_graph(prob, args.steps, args.warmup, stream,
                                                  barrier=barrier, opts=opts)
        launch = (f"CUDA graph of the {args.steps} timed steps, replayed {reps} times back to back "
                  f"(each replay between its own CUDA events; median replay / steps)")
    clocks = sampler.stop(window) if sampler else None
    if not unfused:
        # the same steps launched one by one from the host, for comparison
        ms_loop, _ = time_steps(prob, args.steps, 0, stream, opts=opts, barrier=barrier)
    ms = slowest_rank(dist, ms, dev)
    ms_loop = slowest_rank(dist, ms_loop, dev)
    e2e_ms, h2d, d2h = e2e_steps(prob, max(3, min(args.steps, 20)), stream)
    e2e_ms = slowest_rank(dist, e2e_ms, dev)
    assert fg.fgemm_device_status(stream) == 0
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    pk, pk_src = peaks()
    tflops = w.flops / (ms * 1e-3) / 1e12
    kname = {fg.PATH_TC: "tc_gemm_kernel", fg.PATH_SKINNY: "skinny_kernel",
             fg.PATH_GENERIC: "generic_kernel"}.get(path, "?")
    sustained = window is not None and (window[1] - window[0]) >= SUSTAINED_S
    tpk = tensor_peak(pk, w, sustained)
    hbm_bound = w.unavoidable_bytes() / (pk["hbm_gbs"] * 1e9) > w.flops / (tpk * 1e12)
    if hbm_bound:
        achieved = w.unavoidable_bytes() / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"]}
    else:
        roof = {"bound": "tensor", "achieved": tflops, "peak": tpk, "unit": "TFLOP/s",
                "frac": tflops / tpk}
    which = "sustained" if sustained else "burst"
    roof["peak_source"] = (f"{pk_src} (MEASURED_PEAKS.json bf16 {which}"
                           + (", x 2, the nominal fp8/bf16 ratio)" if w.ab_type == gen.E4M3 else ")")
                           if pk_src == "measured" else pk_src)
    if not hbm_bound:
        roof["frac_of_burst_peak"] = tflops / tensor_peak(pk, w, False)
    roof["traffic"] = recorded_traffic(w.name, kname)
    roof["kernel"] = kname
    cpu = None if args.no_cpu else cpu_baseline(w)
    line = {
        "metric": METRIC, "value": tflops * world, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": gen.TYPE_NAMES[w.ab_type],
        "data": "synthetic (seeded normal inputs, shapes of the workload)",
        "config": {"workload": w.name, "variant": args.variant, "M": w.M, "N": w.N, "K": w.K,
                   "epilogue": w.epilogue,
                   "out": gen.TYPE_NAMES[w.out_type], "bias": gen.TYPE_NAMES[w.bias_type],
                   "path": fg.PATH_NAMES.get(path, str(path)), "plan": prob.plan(opts),
                   "opts": opts,
                   "parallelism": f"replicas{world}", "launch": launch,
                   "stream_loop_ms_per_step": ms_loop,
                   "l2": f"inputs rotate over {len(prob.sets)} sets of {prob.set_bytes / 1e6:.1f} MB "
                         f"(> 2 x L2 {l2 / 1e6:.0f} MB)"},
        "pct_of_peak": 100.0 * tflops / pk["bf16_tflops"],
        "roofline": roof,
        "e2e": {"value": w.flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * reps * ((3 if w.epilogue != "gate" else 2) if unfused else 1),
        "gpu_launches_note": (f"launches of the library's kernels in the timed region: {reps} "
                              f"replays of the {args.steps} steps"),
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle (fp64 CPU) as the reference arm: each step is a bounded row sample."""
    rank, world, _ = env_rank()
    if rank != 0:
        return
    import oracle
    from gemm_epilogue_gb300 import inputs as gen
    oracle.build()
    w = gen.WORKLOADS[args.workload]
    x = gen.make(w)
    threads = oracle.default_threads()
    # 64 rows per thread per step: the oracle's per-call set-up (it decodes B once per call) is
    # then a small part of a step, as in the cpu_baseline leg, which times one larger sample
    rows = max(1, min(w.M, 64 * threads))
    sel = np.arange(rows, dtype=np.int64)
    epi = oracle.EPI_GATE if w.epilogue == "gate" else oracle.EPI_RELU

    def step():
        oracle.gemm_epilogue(x.A, x.B, x.bias, w.M, w.N, w.K, w.ab_type, w.bias_type,
                             w.out_type, epi, Y=x.Y, rows=sel, threads=threads, want_ref=False,
                             y_type=w.y_type)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    tflops = 2.0 * rows * w.N * w.K / dt / 1e12
    sample = f"{rows} of {w.M} output rows of {w.name} per step (all {w.N} columns, K={w.K})"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded normal inputs, shapes of the workload)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": w.epilogue},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_sweep(args):
    """Every workload: fused TFLOP/s, GB/s, roofline fraction; unfused chain; GROUP sweep."""
    import torch
    from gemm_epilogue_gb300 import build as libbuild
    from gemm_epilogue_gb300 import inputs as gen
    libbuild.build()
    import gemm_epilogue_gb300.binding as fg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_DEFAULT
    pk, pk_src = peaks()
    stream = torch.cuda.Stream(device=dev)
    names = args.sweep_workloads.split(",") if args.sweep_workloads else list(gen.WORKLOADS)
    results = []
    for name in names:
        w = gen.WORKLOADS[name]
        unf = w.name in ("square_4096", "glu_gate_1024x21568x4096")
        prob = Problem(w, dev, l2, with_unfused=unf)
        steps = max(5, min(200, int(2e-1 / max(w.flops / 1.2e15, 1e-6))))
        if w.name.startswith("ffn"):
            variants = [{"group_m": g} for g in (1, 4, 8, 16)]
        elif w.name.startswith("skinny"):
            variants = [None] + [{"split_k": s, "skinny_tiles": t}
                                 for t in (1, 2) for s in (2, 4, 8)]
        else:
            variants = [None, {"tail_split": 1}, {"cta_pair": 1}, {"cta_pair": 1, "tail_split": 1},
                        {"bias_init": 1}, {"bias_init": 2}]
        if args.sweep_variants:
            variants = json.loads(args.sweep_variants)
        # Every variant is timed from a cool start: a second of back-to-back load lowers the SM
        # clock (power cap) for a while after it ends, which would bias whichever variant came
        # next.  So the half-second sustained timing of the defaults runs after all the short
        # timings of the workload, and a pause follows every timing.
        sustained = None
        for opts in variants:
            time.sleep(args.sweep_cooldown)
            g = (opts or {}).get("group_m")
            try:
                prob.plan(opts)
            except fg.FgemmError as e:  # a variant the shape cannot take
                print(json.dumps({"workload": name, "opts": opts, "skipped": str(e)}), file=sys.stderr)
                continue
            ms_stream, path = time_steps(prob, steps, 5, stream, opts=opts)
            ms = time_graph(prob, min(steps, 50), 3, stream, opts=opts)
            t = w.flops / (ms * 1e-3) / 1e12
            gbs = w.unavoidable_bytes() / (ms * 1e-3) / 1e9
            t_roof = max(w.flops / (tensor_peak(pk, w) * 1e12), w.unavoidable_bytes() / (pk["hbm_gbs"] * 1e9))
            r = {"workload": name, "opts": opts or "auto", "plan": prob.plan(opts),
                 "path": fg.PATH_NAMES.get(path), "us": ms * 1e3, "us_stream_loop": ms_stream * 1e3,
                 "tflops": t, "gbs": gbs, "roofline_frac": t_roof / (ms * 1e-3),
                 "pct_bf16_peak": 100 * t / pk["bf16_tflops"], "pct_hbm": 100 * gbs / pk["hbm_gbs"]}
            if opts is None:
                sustained = r
            results.append(r)
            print(json.dumps(r), file=sys.stderr, flush=True)
        if sustained is not None:  # the defaults also as the bench line times them: half a second
            time.sleep(args.sweep_cooldown)
            ms_s, _, reps, _ = time_steps_graph(prob, min(steps, 20), 3, stream, opts=None,
                                                 min_seconds=0.5)
            sustained["us_sustained"] = ms_s * 1e3
            sustained["roofline_frac_sustained"] = max(
                w.flops / (tensor_peak(pk, w, True) * 1e12),
                w.unavoidable_bytes() / (pk["hbm_gbs"] * 1e9)) / (ms_s * 1e-3)
            print(json.dumps({"workload": name, "us_sustained": sustained["us_sustained"]}),
                  file=sys.stderr, flush=True)
            time.sleep(2 * args.sweep_cooldown)
        if unf:
            ms, _ = time_steps(prob, steps, 3, stream, unfused=True)
            r = {"workload": name, "variant": "unfused", "us": ms * 1e3,
                 "tflops": w.flops / (ms * 1e-3) / 1e12}
            results.append(r)
            print(json.dumps(r), file=sys.stderr, flush=True)
        assert fg.fgemm_device_status(stream) == 0
        del prob
        torch.cuda.empty_cache()
        if args.sweep_cpu:  # the fp64 oracle on the host cores, a bounded row sample (~2 s)
            r = dict(cpu_baseline(w, target_s=2.0), workload=name, variant="cpu_oracle")
            results.append(r)
            print(json.dumps(r), file=sys.stderr, flush=True)
    if args.sweep_out:  # the whole sweep as one JSON document
        d = os.path.dirname(os.path.abspath(args.sweep_out))
        os.makedirs(d, exist_ok=True)
        with open(args.sweep_out, "w") as f:
            json.dump({"peaks": pk, "peak_source": pk_src, "results": results}, f, indent=1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="square_4096")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--variant", default="fused", choices=["fused", "unfused"],
                    help="unfused: time the GEMM -> elementwise chain instead (traffic comparison)")
    ap.add_argument("--opts", default="",
                    help="fgemm_opts for the timed calls, as JSON (e.g. '{\"group_m\": 8}')")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-workloads", default="")
    ap.add_argument("--sweep-out", default="",
                    help="also write the sweep's results as one JSON file at this path")
    ap.add_argument("--sweep-cpu", action="store_true",
                    help="also time the fp64 oracle on a bounded sample of every swept workload")
    ap.add_argument("--sweep-cooldown", type=float, default=1.0,
                    help="seconds of idle GPU before each sweep timing (clock recovery)")
    ap.add_argument("--sweep-variants", default="",
                    help='JSON list of fgemm_opts dicts (null = defaults) replacing the sweep\'s own')
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
