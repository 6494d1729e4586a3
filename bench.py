#!/usr/bin/env python3
"""Reduction throughput on GB300: GB/s and fraction of measured HBM peak.

One step is one pass of the whole reduction path over one batch of
synthetic inputs resident in HBM:

  x_sum  = 2^30 binary16 values, uniform on [-1, 1), seed 4     (2 GiB)
  x_rows = 65536 x 4096 binary16 values, N(0, 1), seed 2        (512 MiB)
  tcr_reduce_sum(x_sum)   in MMA_CHAIN, FIXED_ORDER, SHUFFLE_TREE, MMA_CHAIN_TMEM
  tcr_reduce_rows(x_rows) in MMA_CHAIN, FIXED_ORDER, SHUFFLE_TREE, MMA_CHAIN_TMEM
  (MMA_CHAIN_TMEM: the tcgen05 / tensor-memory form of MMA_CHAIN)

``value`` is the algorithmic bytes of a step (2 bytes read per input plus
4 bytes written per result) times the steps of all ranks, over the slowest
rank's device time (CUDA events on the launching stream, around all steps
and nothing between the calls: the library launches each call's first
kernel as a programmatic dependent of the kernel before it, which an event
between the two would serialise).  Per call, ``us`` is the average of the
call repeated back to back between two events, ``us_isolated_median`` the
median with events around each call.  Both inputs are far larger than the
129 MB L2, so no flush is needed between calls.

The same JSON line also carries the other configurations of the workload
(``configs``): the 2^20 binary16 sum (L2 flushed before every call by
writing 640 MiB and then reading 256 MiB, outside the timed events; median
of at least 20 calls), the R x block sweep on 2^28 values in [0, 1), and the
2^29 bfloat16 cancellation sum; the read ceiling of the GPU (the best of a
grid sweep of a read-only probe kernel over the 2 GiB input), against which
every fraction is also given; and the oracle on the host cores, all cores
and one.

``--impl reference`` times the CPU oracle instead (the reference arm),
on a bounded sample of the same workload.  ``--sweep`` prints one line per
(R, block) point of the MMA_CHAIN sweep on 2^28 values in [0, 1).
Multi-GPU: every rank runs the same workload on its own GPU (replicas; the
path has no exchange step), one process per GPU under torchrun.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "reduction GB/s and % of GB300 HBM peak (2^30 fp16 sum; 65536×4096 rows)"
UNIT = "GB/s"
N_SUM = 1 << 30
ROWS, COLS = 65536, 4096
WORKLOAD = ("sum of 2^30 fp16 U[-1,1) seed 4 + rows 65536x4096 fp16 N(0,1) seed 2, each in"
            " MMA_CHAIN, FIXED_ORDER, SHUFFLE_TREE and MMA_CHAIN_TMEM")
FALLBACK_HBM_GBS = 6800.0

# kernel launched by each call (the first, reduction launch)
KERNEL_OF = {
    "sum/MMA_CHAIN": "mma_chunk_kernel",
    "sum/FIXED_ORDER": "fixed_chunk_kernel",
    "sum/SHUFFLE_TREE": "shuffle_block_kernel",
    "rows/MMA_CHAIN": "mma_rows_warp_kernel",
    "rows/FIXED_ORDER": "fixed_rows_warp_kernel",
    "rows/SHUFFLE_TREE": "shuffle_rows_warp_kernel",
    "sum/MMA_CHAIN_TMEM": "mma_tmem_kernel",
    "rows/MMA_CHAIN_TMEM": "mma_tmem_rows_flat_kernel",
}


# ------------------------------------------------------------ process setup

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)


def max_over_ranks(value: float, world: int) -> float:
    """The largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_gbps(bytes_per_step: float, steps: int, world: int, seconds: float) -> float:
    """Aggregate GB/s of all ranks: every rank moves bytes_per_step per step."""
    return bytes_per_step * steps * world / seconds / 1e9


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# source file of each kernel; a recorded DRAM traffic figure is stale once
# that file or the shared device headers (helpers, work-split constants,
# warp stream) change
KERNEL_SOURCE = {
    "mma_chunk_kernel": "k_mma.cu", "mma_rows_warp_kernel": "k_mma.cu",
    "fixed_chunk_kernel": "k_fixed.cu", "fixed_rows_warp_kernel": "k_fixed.cu",
    "shuffle_block_kernel": "k_shuffle.cu", "shuffle_rows_warp_kernel": "k_shuffle.cu",
    "combine_kernel": "k_combine.cu", "mma_tmem_kernel": "k_tc05.cu",
    "mma_tmem_rows_kernel": "k_tc05.cu", "mma_tmem_rows_flat_kernel": "k_tc05.cu",
    "gemm_splitk_kernel": "k_gemm.cu",
}
# headers a kernel's source includes beyond the shared device headers
KERNEL_HEADERS = {"k_tc05.cu": ("tc05.cuh",), "k_gemm.cu": ("tc05.cuh",)}


def source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "arithmetic_reduction_tensor_gb300", "csrc")
    src = KERNEL_SOURCE[kernel]
    for f in ("common.cuh", "config.cuh", "stream.cuh") + KERNEL_HEADERS.get(src, ()) + (src,):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel sources (a line 'traffic <kernel> <bytes> <hash>')."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    want = source_hash(kernel)
    for name in sorted(os.listdir(d)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(d, name)) as f:
            for line in f:
                parts = line.strip().strip("`").split()
                if len(parts) == 4 and parts[0] == "traffic" and parts[1] == kernel:
                    if parts[3] == want:
                        return float(parts[2])
    return None


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the work runs."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_csv(lines, self.uuid) or out
        return out


def parse_clock_csv(lines, uuid=None):
    """Median SM clock, max clock and the throttle reasons seen, from
    nvidia-smi CSV lines (noheader, nounits) of ClockSampler.FIELDS."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        p = [c.strip() for c in line.split(",")]
        if len(p) < 10 or (uuid and uuid not in p[1]):
            continue
        try:
            sm.append(float(p[2]))
            smax.append(float(p[3]))
        except ValueError:
            continue
        for name, flag in zip(names, p[6:10]):
            if flag.lower() == "active":
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
            "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ workload

def make_inputs(device):
    import torch
    from arithmetic_reduction_tensor_gb300 import synth
    xs = synth.generate(N_SUM, "uniform_pm1", synth.F16, seed=4)
    xr = synth.generate(ROWS * COLS, "normal", synth.F16, seed=2)
    x_sum = torch.from_numpy(xs.view(np.int16)).to(device)
    x_rows = torch.from_numpy(xr.view(np.int16)).to(device).view(ROWS, COLS)
    return xs, xr, x_sum, x_rows


def build_calls(x_sum, x_rows):
    """[(name, fn(), algorithmic bytes, kernel launches)] for one step."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    dev = x_sum.device
    outs = torch.empty(4 + 4 * ROWS, dtype=torch.float32, device=dev)
    calls = []
    for i, kind in enumerate((tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE)):
        m = tcr.Mode(kind)
        name = "sum/" + tcr.KIND_NAMES[kind]
        o = outs[i:i + 1]
        d = tcr.tcr_order_descriptor(n=N_SUM, mode=m)
        calls.append((name, (lambda m=m, o=o: tcr.tcr_reduce_sum(x_sum, m, out=o)),
                      2 * N_SUM + 4, d["launches"]))
    for i, kind in enumerate((tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE)):
        m = tcr.Mode(kind)
        name = "rows/" + tcr.KIND_NAMES[kind]
        o = outs[3 + i * ROWS:3 + (i + 1) * ROWS]
        d = tcr.tcr_order_descriptor(rows=ROWS, cols=COLS, mode=m)
        calls.append((name, (lambda m=m, o=o: tcr.tcr_reduce_rows(x_rows, m, out=o)),
                      2 * ROWS * COLS + 4 * ROWS, d["launches"]))
    # the tensor-core method once more, on the fifth-generation tensor cores
    m = tcr.Mode(tcr.MMA_CHAIN_TMEM)
    d = tcr.tcr_order_descriptor(n=N_SUM, mode=m)
    o = outs[3 + 3 * ROWS:4 + 3 * ROWS]
    calls.append(("sum/MMA_CHAIN_TMEM", (lambda m=m, o=o: tcr.tcr_reduce_sum(x_sum, m, out=o)),
                  2 * N_SUM + 4, d["launches"]))
    d = tcr.tcr_order_descriptor(rows=ROWS, cols=COLS, mode=m)
    o = outs[4 + 3 * ROWS:4 + 4 * ROWS]
    calls.append(("rows/MMA_CHAIN_TMEM", (lambda m=m, o=o: tcr.tcr_reduce_rows(x_rows, m, out=o)),
                  2 * ROWS * COLS + 4 * ROWS, d["launches"]))
    return calls, outs


def time_device(calls, steps: int, warmup: int, world: int):
    """The timed region: `steps` steps of every call, back to back, with CUDA
    events only around the whole region (an event between two calls would
    hold the next call's launch until the previous one has finished, which
    the library's programmatic dependent launches otherwise overlap).
    Then, per call: the same call `steps` times back to back between two
    events (its average duration, launches overlapped as in a step), and
    `steps` times with events around each call (the median of isolated
    calls)."""
    import torch
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(warmup):
        for _, fn, _, _ in calls:
            fn()
    t0, t1 = ev(), ev()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(steps):
        for _, fn, _, _ in calls:
            fn()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    total_s = t0.elapsed_time(t1) / 1e3
    per_call_avg_ms, per_call_ms = [], []
    for _, fn, _, _ in calls:
        for _ in range(3):
            fn()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        pairs = [(ev(), ev()) for _ in range(steps)]
        for e0, e1 in pairs:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        per_call_avg_ms.append(a.elapsed_time(b) / steps)
        per_call_ms.append([e0.elapsed_time(e1) for e0, e1 in pairs])
    return total_s, per_call_avg_ms, per_call_ms


def time_e2e(xs, xr, calls_factory, steps: int, world: int):
    """Each step: pinned host -> device copy of both inputs, the six calls,
    device -> host copy of every result; CUDA events around all of it.
    The rows input is copied on a second stream while the three sum calls
    run (the calls only wait for the input they read)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    h_sum = torch.from_numpy(xs.view(np.int16)).pin_memory()
    h_rows = torch.from_numpy(xr.view(np.int16)).pin_memory()
    d_sum = torch.empty_like(h_sum, device=dev)
    d_rows = torch.empty_like(h_rows, device=dev).view(ROWS, COLS)
    calls, outs = calls_factory(d_sum, d_rows)
    h_out = torch.empty(outs.numel(), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()

    def step():
        d_sum.copy_(h_sum, non_blocking=True)
        copy_stream.wait_stream(stream)          # previous step's rows calls are done
        with torch.cuda.stream(copy_stream):
            d_rows.view(-1).copy_(h_rows, non_blocking=True)
        sums = [c for c in calls if c[0].startswith("sum/")]
        rows_calls = [c for c in calls if c[0].startswith("rows/")]
        for _, fn, _, _ in sums:
            fn()
        stream.wait_stream(copy_stream)
        for _, fn, _, _ in rows_calls:
            fn()
        h_out.copy_(outs, non_blocking=True)

    step()
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    h2d = h_sum.numel() * 2 + h_rows.numel() * 2
    d2h = h_out.numel() * 4
    return t0.elapsed_time(t1) / 1e3, h2d, d2h


def read_ceiling(x):
    """Best GB/s of the read-only probe kernel (tcr_read_probe) over the
    bytes of x, across grid shapes; median of 10 launches per shape."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    nbytes = x.numel() * x.element_size()
    out = torch.empty(1, dtype=torch.int32, device=x.device)
    best = None
    for block in (256, 512, 1024):
        for ctas in (-1, 1, 2, 4, 8):          # -1: one CTA per chunk of 8 x block vectors
            if block * ctas > 2048:
                continue
            us = timed_median_us(lambda: tcr.tcr_read_probe(x, ctas, block, out=out), 10, 2)
            gbps = nbytes / us / 1e3
            if best is None or gbps > best["gbps"]:
                best = {"gbps": round(gbps, 1), "ctas_per_sm": ctas, "block": block}
    best.update({"bytes": nbytes, "kernel": "read_probe_kernel",
                 "how": "16-byte streaming loads, 8 in flight per thread, XOR of the words; "
                        "best grid shape (1-8 resident CTAs per SM striding over the input, or one "
                        "CTA per chunk: ctas_per_sm -1), median of 10 launches each, queued back to back"})
    return best


def timed_median_us(fn, iters: int, warmup: int, before=None):
    """Median device time of fn() in microseconds (CUDA events around each
    call on the current stream).  Without before(), the calls are queued
    back to back and synchronised once, so the GPU never waits for the
    host between them; before() (an L2 flush) runs ahead of each call,
    outside its events, and keeps the GPU busy while the call is queued."""
    import torch
    for _ in range(warmup):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    torch.cuda.synchronize()
    for e0, e1 in ev:
        if before is not None:
            before()
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)


def time_configs(args, device, ceiling_gbps: float):
    """The workload's other configurations, each call timed alone:
    the 2^20 binary16 sum (seed 0) with L2 flushed before every call; the
    MMA_CHAIN R x block sweep and SHUFFLE_TREE / FIXED_ORDER by block on 2^28
    values in [0, 1) (seed 1); the 2^29 bfloat16 sum of +-2^e (seed 3)."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    from arithmetic_reduction_tensor_gb300 import synth
    peak, _ = load_peaks()
    iters = max(20, min(args.steps, 50))
    out = torch.empty(1, dtype=torch.float32, device=device)
    launches = 0

    def entry(nbytes, us, mode, n):
        nonlocal launches
        launches += (iters + 3) * tcr.tcr_order_descriptor(n=n, mode=mode)["launches"]
        gbps = nbytes / us / 1e3
        return {"us": round(us, 2), "gbps": round(gbps, 1), "frac": round(gbps / peak, 4),
                "frac_of_read_ceiling": round(gbps / ceiling_gbps, 4)}

    res = {}
    # 2^20: 2 MiB, resident in L2 unless flushed.  Writing 640 MiB (about 5x
    # L2) evicts it; reading 256 MiB afterwards replaces the dirty lines that
    # write leaves with clean ones, so the timed call does not wait behind
    # their write-back.  The flush keeps the GPU busy while the call is
    # enqueued, so the events see device time only.
    n1 = 1 << 20
    x1 = torch.from_numpy(synth.generate(n1, "uniform_pm1", synth.F16, seed=0).view(np.int16)).to(device)
    wbuf = torch.empty(640 << 18, dtype=torch.float32, device=device)
    rbuf = torch.ones(1 << 26, dtype=torch.float32, device=device)

    def flush():
        wbuf.zero_()
        rbuf.sum()

    c1 = {}
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN_TMEM):
        m = tcr.Mode(kind, R=4 if kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM) else 0)
        us = timed_median_us(lambda m=m: tcr.tcr_reduce_sum(x1, m, out=out), iters, 3, flush)
        c1[tcr.KIND_NAMES[kind]] = entry(2 * n1 + 4, us, m, n1)
        c1[tcr.KIND_NAMES[kind]]["launches"] = tcr.tcr_order_descriptor(n=n1, mode=m)["launches"]
    res["sum_2p20_f16"] = {"input": "2^20 fp16 U[-1,1) seed 0", "calls": c1,
                           "l2": "flushed before every call: 640 MiB written, then 256 MiB read, "
                                 "outside the timed events",
                           "statistic": f"median of {iters}"}
    del x1, wbuf, rbuf
    torch.cuda.empty_cache()

    n2 = 1 << 28
    x2 = torch.from_numpy(synth.generate(n2, "uniform01", synth.F16, seed=1).view(np.int16)).to(device)
    points = [(tcr.SHUFFLE_TREE, 0, b) for b in (32, 128, 256, 1024)]
    points += [(tcr.FIXED_ORDER, 0, b) for b in (32, 128, 256, 1024)]
    points += [(tcr.MMA_CHAIN, R, b) for R in (1, 2, 4, 5) for b in (32, 128, 256, 1024)]
    points += [(tcr.MMA_CHAIN_TMEM, R, 0) for R in (1, 2, 4, 5, 8)]
    sweep = []
    for kind, R, b in points:
        m = tcr.Mode(kind, R=R, block_threads=b)
        us = timed_median_us(lambda m=m: tcr.tcr_reduce_sum(x2, m, out=out), iters, 3)
        e = entry(2 * n2 + 4, us, m, n2)
        e.update({"kind": tcr.KIND_NAMES[kind], "R": R, "block": b})
        sweep.append(e)
    res["sum_2p28_f16_sweep"] = {"input": "2^28 fp16 U[0,1) seed 1, 512 MiB (larger than L2)",
                                 "points": sweep, "statistic": f"median of {iters}"}
    del x2
    torch.cuda.empty_cache()

    n4 = 1 << 29
    x4 = torch.from_numpy(synth.generate(n4, "pow2", synth.BF16, seed=3).view(np.int16)).to(device)
    c4 = {}
    for kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        m = tcr.Mode(kind, dtype=tcr.BF16)
        us = timed_median_us(lambda m=m: tcr.tcr_reduce_sum(x4, m, out=out), iters, 3)
        c4[tcr.KIND_NAMES[kind]] = entry(2 * n4 + 4, us, m, n4)
    res["sum_2p29_bf16"] = {"input": "2^29 bf16 +-2^e, e in [-20, 10], seed 3, 1 GiB", "calls": c4,
                            "statistic": f"median of {iters}"}
    del x4
    torch.cuda.empty_cache()
    res["launches"] = launches
    return res


# ------------------------------------------------------------ CPU oracle

def oracle_pass(xs_sample, xr_sample, threads: int):
    """The oracle's work for one step of the workload, on a sample:
    what each of the six calls is checked against."""
    import oracle
    from tests import spec
    oracle.exact_sum(xs_sample, oracle.F16, threads)
    oracle.fixed_order(xs_sample, oracle.F16, threads)
    oracle.shuffle_tree(xs_sample, oracle.F16, *spec.shuffle_team(xs_sample.size), threads=threads)
    oracle.exact_sum_rows(xr_sample, oracle.F16, threads)
    oracle.fixed_order_rows(xr_sample, oracle.F16, threads)
    oracle.shuffle_tree_rows(xr_sample, oracle.F16, *spec.shuffle_team(COLS), threads=threads)
    return 3 * 2 * xs_sample.size + 3 * (2 * xr_sample.size + 4 * xr_sample.shape[0])


def cpu_samples(xs, xr, budget_s: float, threads: int):
    """Sizes the sample so one oracle pass takes about budget_s seconds."""
    n0, r0 = 1 << 22, 1 << 10
    t = time.perf_counter()
    oracle_pass(xs[:n0], xr[:r0 * COLS].reshape(r0, COLS), threads)
    dt = max(time.perf_counter() - t, 1e-3)
    scale = max(1.0, budget_s / dt)
    n = int(min(xs.size, n0 * scale))
    r = int(min(xr.size // COLS, r0 * scale))
    return xs[:n], xr[:r * COLS].reshape(r, COLS)


def cpu_baseline(xs, xr, budget_s: float = 10.0):
    """The oracle on all host cores and on one, each on a sample sized for
    about budget_s seconds."""
    import oracle
    legs = []
    for threads in (oracle.default_threads(), 1):
        s, r = cpu_samples(xs, xr, budget_s, threads)
        t = time.perf_counter()
        nbytes = oracle_pass(s, r, threads)
        dt = time.perf_counter() - t
        legs.append({"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": threads,
                     "kind": "oracle",
                     "sample": f"first {s.size} of the 2^30 sum inputs and first {r.shape[0]} of the "
                               f"65536 rows; exact sum, fixed-order tree and shuffle-tree emulation of each",
                     "seconds": round(dt, 3)})
    line = legs[0]
    line["single_thread"] = legs[1]
    return line


# ------------------------------------------------------------ arms

def reference_arm(args):
    """The oracle timed as the reference arm, on a bounded sample per step."""
    import oracle
    from arithmetic_reduction_tensor_gb300 import synth
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    threads = oracle.default_threads()
    budget = max(0.05, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    n_probe = 1 << 26
    xs = synth.generate(n_probe, "uniform_pm1", synth.F16, seed=4)
    xr = synth.generate(4096 * COLS, "normal", synth.F16, seed=2)
    s, r = cpu_samples(xs, xr.reshape(-1), budget, threads)
    for _ in range(args.warmup):
        oracle_pass(s, r, threads)
    t = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_pass(s, r, threads)
    dt = time.perf_counter() - t
    value = nbytes / dt / 1e9
    sample = (f"per step: first {s.size} of the 2^30 sum inputs and first {r.shape[0]} of the "
              f"65536 rows; exact sum, fixed-order tree and shuffle-tree emulation of each")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def sweep_arm(args):
    """MMA_CHAIN R x block sweep against SHUFFLE_TREE and FIXED_ORDER on 2^28
    values in [0, 1), and MMA_CHAIN_TMEM by R (its CTA shape is fixed)."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    from arithmetic_reduction_tensor_gb300 import synth
    torch.cuda.set_device(0)
    n = 1 << 28
    x = torch.from_numpy(synth.generate(n, "uniform01", synth.F16, seed=1).view(np.int16)).cuda()
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    peak, _ = load_peaks()
    points = [(tcr.SHUFFLE_TREE, 0, b) for b in (32, 128, 256, 1024)]
    points += [(tcr.FIXED_ORDER, 0, b) for b in (32, 128, 256, 1024)]
    points += [(tcr.MMA_CHAIN, R, b) for R in (1, 2, 4, 5) for b in (32, 128, 256, 1024)]
    points += [(tcr.MMA_CHAIN_TMEM, R, 0) for R in (1, 2, 4, 5, 8)]
    for kind, R, b in points:
        m = tcr.Mode(kind, R=R, block_threads=b)
        for _ in range(3):
            tcr.tcr_reduce_sum(x, m, out=out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            tcr.tcr_reduce_sum(x, m, out=out)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        gbps = 2 * n / us / 1e3
        print(json.dumps({"sweep": "sum 2^28 fp16 U[0,1) seed 1", "kind": tcr.KIND_NAMES[kind],
                          "R": R, "block": b, "us": round(us, 2), "gbps": round(gbps, 1),
                          "frac": round(gbps / peak, 4)}), flush=True)
    return 0


def profile_arm(args):
    """A small case for ncu: each sum mode once on 2^28 fp16 values (512 MiB,
    larger than L2), each rows mode once on 32768 x 4096 rows (256 MiB), and
    the tcgen05 MMA_CHAIN sum and rows.  ``--profile-case f32``: the same
    bytes in binary32 (2^27 sum, 32768 x 2048 rows), the three mma.sync-era
    modes.  ``--profile-case gemm``: the split-K GEMM on 4096^3 (one split)
    and 1024 x 1024 x 16384 (the default split).  ``--profile-case short``:
    the packed short-row kernels, each mode once on 4194304 x 64 fp16 rows
    (512 MiB) and once on 2684354 x 100 (rows not 16-byte aligned).
    ``--profile-case odd``: FIXED_ORDER and MMA_CHAIN on rows of odd length
    (536334 x 1001 and 1046502 x 513 fp16, every other row on a 2-byte
    boundary).  ``--profile-case blocked``: FIXED_ORDER's blocked order on
    the 2^28 fp16 sum with runs of 256 and on 32768 x 4096 rows with runs of
    32 and 256."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    from arithmetic_reduction_tensor_gb300 import synth
    torch.cuda.set_device(0)
    if args.profile_case == "gemm":
        gen = torch.Generator(device="cuda").manual_seed(5)
        for M, N, K, S in ((4096, 4096, 4096, 1), (1024, 1024, 16384, 0)):
            A = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
            W = torch.randn(N, K, device="cuda", generator=gen).to(torch.bfloat16)
            for _ in range(args.steps):
                tcr.tcr_gemm_splitk(A, W, splits=S)
        torch.cuda.synchronize()
        print("profile case done", flush=True)
        return 0
    if args.profile_case == "short":
        n = 1 << 28
        x = torch.from_numpy(synth.generate(n, "normal", synth.F16, seed=2).view(np.int16)).cuda()
        shapes = ((n // 64, 64), (n // 100, 100))
        for _ in range(args.steps):
            for rows, cols in shapes:
                for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
                    tcr.tcr_reduce_rows(x[:rows * cols].view(rows, cols), tcr.Mode(kind))
        torch.cuda.synchronize()
        print("profile case done", flush=True)
        return 0
    if args.profile_case == "odd":
        n = 1 << 29
        x = torch.from_numpy(synth.generate(n, "normal", synth.F16, seed=2).view(np.int16)).cuda()
        shapes = ((n // 1001, 1001), (n // 513, 513))
        for _ in range(args.steps):
            for rows, cols in shapes:
                for kind in (tcr.FIXED_ORDER, tcr.MMA_CHAIN):
                    tcr.tcr_reduce_rows(x[:rows * cols].view(rows, cols), tcr.Mode(kind))
        torch.cuda.synchronize()
        print("profile case done", flush=True)
        return 0
    if args.profile_case == "blocked":
        x = torch.from_numpy(synth.generate(1 << 28, "uniform_pm1", synth.F16, seed=4).view(np.int16)).cuda()
        r = torch.from_numpy(synth.generate(32768 * COLS, "normal", synth.F16, seed=2).view(np.int16))
        r = r.cuda().view(32768, COLS)
        for _ in range(args.steps):
            tcr.tcr_reduce_sum(x, tcr.Mode(tcr.FIXED_ORDER, run_log2=8))
            tcr.tcr_reduce_rows(r, tcr.Mode(tcr.FIXED_ORDER, run_log2=5))
            tcr.tcr_reduce_rows(r, tcr.Mode(tcr.FIXED_ORDER, run_log2=8))
        torch.cuda.synchronize()
        print("profile case done", flush=True)
        return 0
    if args.profile_case == "f32":
        x = torch.from_numpy(synth.generate(1 << 27, "uniform_pm1", synth.F32, seed=4).view(np.float32))
        r = torch.from_numpy(synth.generate(32768 * 2048, "normal", synth.F32, seed=2).view(np.float32))
        x, r = x.cuda(), r.cuda().view(32768, 2048)
        for _ in range(args.steps):
            for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
                tcr.tcr_reduce_sum(x, tcr.Mode(kind, dtype=tcr.F32))
                tcr.tcr_reduce_rows(r, tcr.Mode(kind, dtype=tcr.F32))
        torch.cuda.synchronize()
        print("profile case done", flush=True)
        return 0
    n = 1 << 28
    x = torch.from_numpy(synth.generate(n, "uniform_pm1", synth.F16, seed=4).view(np.int16)).cuda()
    r = torch.from_numpy(synth.generate(32768 * COLS, "normal", synth.F16, seed=2).view(np.int16))
    r = r.cuda().view(32768, COLS)
    for _ in range(args.steps):
        for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
            tcr.tcr_reduce_sum(x, tcr.Mode(kind))
            tcr.tcr_reduce_rows(r, tcr.Mode(kind))
        tcr.tcr_reduce_sum(x, tcr.Mode(tcr.MMA_CHAIN_TMEM))
        tcr.tcr_reduce_rows(r, tcr.Mode(tcr.MMA_CHAIN_TMEM))
    torch.cuda.synchronize()
    print("profile case done", flush=True)
    return 0


def extras_arm(args):
    """Beyond the hot path, one JSON line per call: the sum of squares (2^30
    sum and 65536 x 4096 rows, every mode), binary32 inputs (2^29 sum and
    65536 x 2048 rows -- the same bytes as the 16-bit workload -- every mode,
    sums and sums of squares), FIXED_ORDER's blocked order (runs of 2^c
    inputs left to right, then the tree) on the 16-bit workload, the
    fused row moments (sum and sum of squares, mean and variance, one pass),
    short rows (views of the 2^30 sum input as rows of 64, 256 and 1024
    inputs, rows of 100 whose starts are not 16-byte aligned, row moments of
    768), long rows of 4095 inputs and the sum from a base one input past a
    16-byte boundary."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    from arithmetic_reduction_tensor_gb300 import synth
    torch.cuda.set_device(0)
    peak, _ = load_peaks()
    xs = torch.from_numpy(synth.generate(N_SUM, "uniform_pm1", synth.F16, seed=4).view(np.int16)).cuda()
    xr = torch.from_numpy(synth.generate(ROWS * COLS, "normal", synth.F16, seed=2).view(np.int16))
    xr = xr.cuda().view(ROWS, COLS)
    out = torch.empty(ROWS, dtype=torch.float32, device="cuda")
    calls = []
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        m = tcr.Mode(kind)
        calls.append(("sum_squares/" + tcr.KIND_NAMES[kind], 2 * N_SUM + 4,
                      lambda m=m: tcr.tcr_reduce_sum_squares(xs, m, out=out[:1])))
        calls.append(("rows_sum_squares/" + tcr.KIND_NAMES[kind], 2 * ROWS * COLS + 4 * ROWS,
                      lambda m=m: tcr.tcr_reduce_rows_sum_squares(xr, m, out=out)))
    n32, cols32 = N_SUM // 2, COLS // 2
    fs = torch.from_numpy(synth.generate(n32, "uniform_pm1", synth.F32, seed=4).view(np.float32)).cuda()
    fr = torch.from_numpy(synth.generate(ROWS * cols32, "normal", synth.F32, seed=2).view(np.float32))
    fr = fr.cuda().view(ROWS, cols32)
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        m = tcr.Mode(kind, dtype=tcr.F32)
        k = tcr.KIND_NAMES[kind]
        calls.append(("f32_sum/" + k, 4 * n32 + 4, lambda m=m: tcr.tcr_reduce_sum(fs, m, out=out[:1])))
        calls.append(("f32_rows/" + k, 4 * ROWS * cols32 + 4 * ROWS,
                      lambda m=m: tcr.tcr_reduce_rows(fr, m, out=out)))
        calls.append(("f32_sum_squares/" + k, 4 * n32 + 4,
                      lambda m=m: tcr.tcr_reduce_sum_squares(fs, m, out=out[:1])))
    # the blocked-sequential-then-tree order (FIXED_ORDER, runs of 2^c)
    for c in (2, 3, 4, 6, 8, 10):
        m = tcr.Mode(tcr.FIXED_ORDER, run_log2=c)
        calls.append((f"blocked_sum/c={c}", 2 * N_SUM + 4,
                      lambda m=m: tcr.tcr_reduce_sum(xs, m, out=out[:1])))
    for c in (3, 5, 8):
        m = tcr.Mode(tcr.FIXED_ORDER, run_log2=c)
        calls.append((f"blocked_rows/c={c}", 2 * ROWS * COLS + 4 * ROWS,
                      lambda m=m: tcr.tcr_reduce_rows(xr, m, out=out)))
    # the fused row moments: sum and sum of squares (and mean/variance) in one pass
    out2 = torch.empty(ROWS, dtype=torch.float32, device="cuda")
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        m = tcr.Mode(kind)
        k = tcr.KIND_NAMES[kind]
        calls.append(("rows_moments/" + k, 2 * ROWS * COLS + 8 * ROWS,
                      lambda m=m: tcr.tcr_reduce_rows_moments(xr, m, sums=out, sums_of_squares=out2)))
        calls.append(("rows_mean_var/" + k, 2 * ROWS * COLS + 8 * ROWS,
                      lambda m=m: tcr.tcr_reduce_rows_mean_var(xr, m, mean=out, var=out2)))
    # short rows (packed several to a warp), unaligned rows and base: views
    # of the sum input, every row its own segment
    kinds4 = (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN_TMEM)
    for cols in (64, 256, 1024):
        v = xs.view(N_SUM // cols, cols)
        o = torch.empty(N_SUM // cols, dtype=torch.float32, device="cuda")
        for kind in kinds4:
            m = tcr.Mode(kind)
            calls.append((f"short_rows_{cols}/" + tcr.KIND_NAMES[kind], 2 * N_SUM + 4 * (N_SUM // cols),
                          lambda m=m, v=v, o=o: tcr.tcr_reduce_rows(v, m, out=o)))
    for cols in (100, 4095):
        nr = N_SUM // cols
        v = xs[:nr * cols].view(nr, cols)
        o = torch.empty(nr, dtype=torch.float32, device="cuda")
        for kind in kinds4:
            m = tcr.Mode(kind)
            calls.append((f"unaligned_rows_{cols}/" + tcr.KIND_NAMES[kind], 2 * nr * cols + 4 * nr,
                          lambda m=m, v=v, o=o: tcr.tcr_reduce_rows(v, m, out=o)))
    xm = xs[1:]
    for kind in kinds4:
        m = tcr.Mode(kind)
        calls.append(("unaligned_sum/" + tcr.KIND_NAMES[kind], 2 * (N_SUM - 1) + 4,
                      lambda m=m: tcr.tcr_reduce_sum(xm, m, out=out[:1])))
    nr768 = N_SUM // 768
    v768 = xs[:nr768 * 768].view(nr768, 768)
    oa = torch.empty(nr768, dtype=torch.float32, device="cuda")
    ob = torch.empty(nr768, dtype=torch.float32, device="cuda")
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        m = tcr.Mode(kind)
        calls.append(("short_rows_768_mean_var/" + tcr.KIND_NAMES[kind], 2 * nr768 * 768 + 8 * nr768,
                      lambda m=m: tcr.tcr_reduce_rows_mean_var(v768, m, mean=oa, var=ob)))
    for name, nbytes, fn in calls:
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        gbps = nbytes / us / 1e3
        print(json.dumps({"extra": name, "us": round(us, 2), "gbps": round(gbps, 1),
                          "frac": round(gbps / peak, 4), "steps": args.steps}), flush=True)
    # small inputs (2^20 fp16, 2 MiB -- launch-bound): each call timed alone
    # after a read of a 256 MiB buffer (which evicts the input from L2 and,
    # unlike a write, leaves no dirty lines whose write-back the call would
    # wait behind); the GPU is busy with that read while the call is enqueued,
    # so the events see device time only
    x20 = xs[:1 << 20]
    flush = torch.ones(1 << 26, dtype=torch.float32, device="cuda")
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN_TMEM):
        m = tcr.Mode(kind)
        for _ in range(args.warmup):
            tcr.tcr_reduce_sum(x20, m, out=out[:1])
        times = []
        for _ in range(args.steps):
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            tcr.tcr_reduce_sum(x20, m, out=out[:1])
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(times)
        print(json.dumps({"extra": "small_sum_2p20/" + tcr.KIND_NAMES[kind], "us": round(us, 2),
                          "gbps": round(2 * (1 << 20) / us / 1e3, 1), "l2": "flushed",
                          "launches": tcr.tcr_order_descriptor(n=1 << 20, mode=m)["launches"],
                          "statistic": "median", "steps": args.steps}), flush=True)
    return 0


def load_bf16_peaks():
    """(burst, sustained) measured bf16 GEMM TFLOP/s and their source."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


def gemm_arm(args):
    """The split-K GEMM with the declared combine: TFLOP/s (2 M N K per call)
    for square shapes at S = 1 and K-heavy shapes at the default S and at
    S = 1.  Per shape: 20 calls back to back (a burst, against the measured
    burst bf16 peak) and `steps` calls back to back (against the measured
    sustained peak: a long run settles under the power limit), clocks
    sampled throughout."""
    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    torch.cuda.set_device(0)
    burst, sustained, src = load_bf16_peaks()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(0).uuid)
    except Exception:
        pass
    gen = torch.Generator(device="cuda").manual_seed(5)
    cases = [(4096, 4096, 4096, 0), (8192, 8192, 8192, 0), (1024, 1024, 16384, 0),
             (1024, 1024, 16384, 1), (512, 512, 32768, 0), (512, 512, 32768, 1)]

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    for M, N, K, S in cases:
        A = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
        W = torch.randn(N, K, device="cuda", generator=gen).to(torch.bfloat16)
        C = torch.empty(M, N, device="cuda")
        d = tcr.tcr_gemm_descriptor(M, N, K, S, tcr.BF16)
        fn = lambda: tcr.tcr_gemm_splitk(A, W, splits=S, out=C)
        for _ in range(args.warmup):
            fn()
        clocks = ClockSampler(uuid)
        clocks.start()
        us_burst = timed(fn, 20)
        us = timed(fn, args.steps)
        clk = clocks.stop()
        tf_burst = 2.0 * M * N * K / us_burst / 1e6
        tf = 2.0 * M * N * K / us / 1e6
        print(json.dumps({"gemm": f"{M}x{N}x{K} bf16", "splits": d["splits"], "k_split": d["k_split"],
                          "tile": [d["tile_m"], d["tile_n"]], "grid": d["launch_grid"],
                          "us_burst": round(us_burst, 2), "tflops_burst": round(tf_burst, 1),
                          "frac_of_burst_peak": round(tf_burst / burst, 4),
                          "us": round(us, 2), "tflops": round(tf, 1),
                          "frac_of_sustained_peak": round(tf / sustained, 4), "steps": args.steps,
                          "peaks": {"burst": burst, "sustained": sustained, "source": src},
                          "clocks": clk}), flush=True)
        del A, W, C
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tcr", "reference"], default="tcr")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--extras", action="store_true",
                    help="time the sum of squares and binary32 calls (beyond the hot path) and exit")
    ap.add_argument("--profile-case", nargs="?", const="f16", choices=["f16", "f32", "gemm", "short", "odd", "blocked"],
                    default=None,
                    help="run the small ncu case (2^28 sum, 32768 x 4096 rows; f32: the same "
                         "bytes in binary32; gemm: 4096^3 and 1024^2 x 16384 bf16; short: packed "
                         "rows of 64 and 100 fp16) and exit")
    ap.add_argument("--gemm", action="store_true",
                    help="time the split-K GEMM with the declared combine (TFLOP/s) and exit")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: max(3, steps // 40)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank, world, local = dist_info()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 runs under torchrun, one process per GPU")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    from arithmetic_reduction_tensor_gb300.build import build_library

    if args.sweep:
        build_library()
        return sweep_arm(args)
    if args.profile_case:
        build_library()
        return profile_arm(args)
    if args.extras:
        build_library()
        return extras_arm(args)
    if args.gemm:
        build_library()
        return gemm_arm(args)

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    build_library()
    tcr.c_api()
    device = torch.device("cuda", local)
    xs, xr, x_sum, x_rows = make_inputs(device)
    calls, _ = build_calls(x_sum, x_rows)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    total_s, per_call_avg_ms, per_call_ms = time_device(calls, args.steps, args.warmup, world)
    ceiling = read_ceiling(x_sum)
    e2e_steps = args.e2e_steps or max(3, args.steps // 40)
    del x_sum, x_rows, calls
    torch.cuda.empty_cache()
    e2e_s, h2d, d2h = time_e2e(xs, xr, build_calls, e2e_steps, world)
    torch.cuda.empty_cache()
    configs = time_configs(args, device, ceiling["gbps"])
    clk = clocks.stop()

    meta = build_calls_meta()
    bytes_per_step = sum(m[1] for m in meta)
    max_s = max_over_ranks(total_s, world)
    max_e2e = max_over_ranks(e2e_s, world)
    value = whole_job_gbps(bytes_per_step, args.steps, world, max_s)
    e2e_value = whole_job_gbps(bytes_per_step, e2e_steps, world, max_e2e)
    peak, peak_src = load_peaks()

    calls_out = {}
    for (name, nbytes, launches), avg_ms, ms in zip(meta, per_call_avg_ms, per_call_ms):
        avg_us = avg_ms * 1e3
        med_us = statistics.median(ms) * 1e3
        gbps = nbytes / avg_us / 1e3
        calls_out[name] = {"us": round(avg_us, 2), "gbps": round(gbps, 1),
                           "gelem_per_s": round(call_elements(name) / avg_us / 1e3, 1),
                           "frac": round(gbps / peak, 4),
                           "frac_of_read_ceiling": round(gbps / ceiling["gbps"], 4),
                           "us_isolated_median": round(med_us, 2),
                           "launches": launches}
    dom = max(calls_out, key=lambda k: calls_out[k]["us"])
    dom_nbytes = dict((m[0], m[1]) for m in meta)[dom]
    dom_gbps = dom_nbytes / calls_out[dom]["us"] / 1e3
    elements_per_step = sum(call_elements(m[0]) for m in meta)
    launches = sum(m[2] for m in meta) * args.steps

    if rank != 0:
        return 0
    cpu = cpu_baseline(xs, xr, args.cpu_budget) if world == 1 else None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(max_s / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "inputs 2 GiB and 512 MiB, larger than L2; no flush",
                   "input_dtype": "fp16", "accumulate": "fp32", "block_threads": 256,
                   "mma_chain_R": tcr.tcr_order_descriptor(n=N_SUM, mode=tcr.Mode(tcr.MMA_CHAIN))["chain_R"]},
        "frac_of_peak": round(value / world / peak, 4),
        "peak_gbs": peak, "peak_source": peak_src,
        "read_ceiling": ceiling,
        "frac_of_read_ceiling": round(value / world / ceiling["gbps"], 4),
        "gelem_per_s": round(elements_per_step * args.steps * world / max_s / 1e9, 1),
        "calls": calls_out,
        # page 1 reports about 3.2x for its tensor-core reduction over a
        # conventional GPU reduction, on hardware the page does not name
        "mma_chain_over_shuffle_tree": round(calls_out["sum/SHUFFLE_TREE"]["us"] /
                                             calls_out["sum/MMA_CHAIN"]["us"], 3),
        "roofline": {"bound": "hbm", "kernel": KERNEL_OF[dom], "call": dom,
                     "achieved": round(dom_gbps, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dom_gbps / peak, 4), "traffic": recorded_traffic(KERNEL_OF[dom]),
                     "duration": "average of the call repeated back to back between two events "
                                 "(the whole call: reduction + combine launch)",
                     "peak_source": peak_src,
                     "read_ceiling": ceiling["gbps"],
                     "frac_of_read_ceiling": round(dom_gbps / ceiling["gbps"], 4)},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches,
        "configs": configs,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def call_elements(name: str) -> int:
    """Inputs one bench call reduces."""
    return N_SUM if name.startswith("sum/") else ROWS * COLS


def build_calls_meta():
    """(name, algorithmic bytes, launches) of the eight calls of a step."""
    import arithmetic_reduction_tensor_gb300 as tcr
    meta = []
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        d = tcr.tcr_order_descriptor(n=N_SUM, mode=tcr.Mode(kind))
        meta.append(("sum/" + tcr.KIND_NAMES[kind], 2 * N_SUM + 4, d["launches"]))
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        d = tcr.tcr_order_descriptor(rows=ROWS, cols=COLS, mode=tcr.Mode(kind))
        meta.append(("rows/" + tcr.KIND_NAMES[kind], 2 * ROWS * COLS + 4 * ROWS, d["launches"]))
    d = tcr.tcr_order_descriptor(n=N_SUM, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM))
    meta.append(("sum/MMA_CHAIN_TMEM", 2 * N_SUM + 4, d["launches"]))
    d = tcr.tcr_order_descriptor(rows=ROWS, cols=COLS, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM))
    meta.append(("rows/MMA_CHAIN_TMEM", 2 * ROWS * COLS + 4 * ROWS, d["launches"]))
    return meta


if __name__ == "__main__":
    sys.exit(main())
