#!/usr/bin/env python3
"""Benchmark of the collective datapath on one GB300 (or N independent replicas).

One step = one AllReduce (sum) over 8 emulated ranks of 32 Mi bf16 elements
(64 MiB) each, through the library's C ABI: layout, tiling, one persistent
kernel running the N-to-1 reduce Atom, written to all 8 outputs.  The metric
is HBM GB/s counted as algorithmic bytes (every input byte read once, every
output byte written once: 2 * 8 * 64 MiB = 1 GiB per step) over device time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl own|reference]
                  [--workload NAME]

Prints one JSON line (rank 0).  With --impl reference the CPU oracle is timed
on the host cores on a bounded sample of the same workload instead.
--workload picks another of the five workloads' largest cases (ReduceScatter,
AllGather, AllToAll, AllToAllV, AllGatherV) for the same measurement; the
default is the AllReduce above.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORLD = 8
N_ELEMS = 32 << 20          # per rank
ELEM = 2                    # bf16
S = N_ELEMS * ELEM          # bytes per rank
ALGO_BYTES = 2 * WORLD * S  # N inputs read + N outputs written
METRIC = "AllReduce/ReduceScatter/AllGather/AllToAll HBM GB/s vs size, % of GB300 HBM peak"
WORKLOAD = "AllReduce sum, 8 emulated ranks on one GPU, bf16 in/out, fp32 ascending-rank accumulation, " \
           "32 Mi elements (64 MiB) per rank, N(0,1), seed 1"


class Workload:
    """One collective at one workload size: host inputs, output sizes, the call, its bytes."""

    def __init__(self, name, desc, dtype, make_inputs, out_bytes, call, algo_bytes, coll, tune_bytes, tune=None):
        self.name, self.desc, self.dtype = name, desc, dtype
        self.make_inputs, self.out_bytes, self.call = make_inputs, out_bytes, call
        self.algo_bytes, self.coll, self.tune_bytes = algo_bytes, coll, tune_bytes
        self.tune = tune  # tuning override applied to the handle (None: the table's choice)


def workloads(P, inputs, w4_mib=256):
    """The five workloads' largest single-GPU cases (the first is the headline).
    w4_mib: per-rank size of the AllGather / AllToAll byte workloads (256 MiB;
    smaller only for profiler captures, which must stay a few GB)."""
    MI = 1 << 20
    C5, c5 = inputs.w5_counts(WORLD)
    G = w4_mib * MI
    w = [
        Workload("allreduce_bf16_8x64MiB", WORKLOAD, "bf16",
                 lambda: list(inputs.w2_allreduce_bf16(WORLD, N_ELEMS, seed=1)),
                 [S] * WORLD, lambda h, s, d, st: P.purlin_all_reduce(h, s, d, S, P.PL_BF16, 0, st),
                 ALGO_BYTES, P.PL_COLL_ALL_REDUCE, S),
        Workload("allreduce_two_shot_bf16_8x64MiB", WORKLOAD.replace("AllReduce sum", "AllReduce sum, two-shot "
                 "layout (each owner reduces its range, notifies, and the range is copied to the other ranks: "
                 "SNAC between CTAs),", 1), "bf16",
                 lambda: list(inputs.w2_allreduce_bf16(WORLD, N_ELEMS, seed=1)),
                 [S] * WORLD, lambda h, s, d, st: P.purlin_all_reduce(h, s, d, S, P.PL_BF16, 0, st),
                 ALGO_BYTES, P.PL_COLL_ALL_REDUCE, S, tune={"layout": P.PL_LAYOUT_TWO_SHOT}),
        Workload("allreduce_ring_bf16_8x64MiB", WORKLOAD.replace("AllReduce sum", "AllReduce sum, ring layout "
                 "(per tile a binary32 running sum handed from rank to rank in ascending order, then the "
                 "finished tile passed around the ring: 2(N-1) SNAC stages per tile)", 1), "bf16",
                 lambda: list(inputs.w2_allreduce_bf16(WORLD, N_ELEMS, seed=1)),
                 [S] * WORLD, lambda h, s, d, st: P.purlin_all_reduce(h, s, d, S, P.PL_BF16, 0, st),
                 ALGO_BYTES, P.PL_COLL_ALL_REDUCE, S, tune={"layout": P.PL_LAYOUT_RING}),
        Workload("reduce_scatter_f32_8x256MiB",
                 "ReduceScatter sum, 8 ranks, fp32, 64 Mi elements (256 MiB) per rank, U(-1,1), seed 2", "f32",
                 lambda: list(inputs.w3_reduce_scatter(WORLD, 64 * MI, seed=2, dtype="f32")),
                 [32 * MI] * WORLD, lambda h, s, d, st: P.purlin_reduce_scatter(h, s, d, 256 * MI, P.PL_F32, 0, st),
                 WORLD * 256 * MI + 256 * MI, P.PL_COLL_REDUCE_SCATTER, 256 * MI),
        Workload("reduce_scatter_bf16_8x128MiB",
                 "ReduceScatter sum, 8 ranks, bf16, 64 Mi elements (128 MiB) per rank, U(-1,1), seed 2", "bf16",
                 lambda: list(inputs.w3_reduce_scatter(WORLD, 64 * MI, seed=2, dtype="bf16")),
                 [16 * MI] * WORLD, lambda h, s, d, st: P.purlin_reduce_scatter(h, s, d, 128 * MI, P.PL_BF16, 0, st),
                 WORLD * 128 * MI + 128 * MI, P.PL_COLL_REDUCE_SCATTER, 128 * MI),
        Workload("all_gather_u8_8x256MiB", f"AllGather, 8 ranks, uint8 payload, {w4_mib} MiB per rank, seed 3", "u8",
                 lambda: list(inputs.w4_bytes(WORLD, G)),
                 [WORLD * G] * WORLD, lambda h, s, d, st: P.purlin_all_gather(h, s, d, G, st),
                 WORLD * G * (1 + WORLD), P.PL_COLL_ALL_GATHER, G),
        Workload("all_to_all_u8_8x256MiB", f"AllToAll, 8 ranks, uint8 payload, {w4_mib} MiB per rank, seed 3", "u8",
                 lambda: list(inputs.w4_bytes(WORLD, G)),
                 [G] * WORLD, lambda h, s, d, st: P.purlin_all_to_all(h, s, d, G, st),
                 2 * WORLD * G, P.PL_COLL_ALL_TO_ALL, G),
        Workload("all_to_all_v_bf16_w5",
                 "AllToAllV, 8 ranks, bf16 N(0,1), counts uniform in [0, 4 Mi] elements with forced zeros and "
                 "counts not multiple of 8, seed 4", "bf16",
                 lambda: inputs.w5_payloads(C5, c5)[0],
                 [int(C5[:, d].sum()) * 2 for d in range(WORLD)],
                 lambda h, s, d, st: P.purlin_all_to_all_v(h, s, d, [int(v) * 2 for v in C5.reshape(-1)], st),
                 2 * int(C5.sum()) * 2, P.PL_COLL_ALL_TO_ALL_V, int(C5.sum()) * 2 // WORLD),
        Workload("all_gather_v_bf16_w5",
                 "AllGatherV, 8 ranks, bf16 N(0,1), counts uniform in [0, 4 Mi] elements, seed 4", "bf16",
                 lambda: inputs.w5_payloads(C5, c5)[1],
                 [int(c5.sum()) * 2] * WORLD,
                 lambda h, s, d, st: P.purlin_all_gather_v(h, s, d, [int(v) * 2 for v in c5], st),
                 int(c5.sum()) * 2 * (1 + WORLD), P.PL_COLL_ALL_GATHER_V, int(c5.sum()) * 2 // WORLD),
    ]
    return {x.name: x for x in w}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-collective side table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--workload", default="allreduce_bf16_8x64MiB",
                    help="which collective to time (default: the AllReduce headline)")
    ap.add_argument("--device-only", action="store_true",
                    help="time the device leg only: no end-to-end legs, side table or CPU baseline "
                         "(profiler captures: few launches, little memory)")
    ap.add_argument("--tune", default="",
                    help="tuning fields over the workload's own, e.g. store_hint=3,snac_lag=2")
    ap.add_argument("--w4-mib", type=int, default=256,
                    help="per-rank MiB of the AllGather / AllToAll workloads (smaller for profiler captures)")
    args = ap.parse_args()
    if args.device_only:
        args.no_extras = args.no_cpu = True
    return args


# ------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float, device=None) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed work runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def source_hash(files):
    """Hash of the given repository files (the sources a kernel is built from)."""
    h = hashlib.sha256()
    for rel in sorted(files):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(name, tune):
    """DRAM bytes per launch of the workload's kernel from the committed ncu summary,
    or None when the kernel changed since the counters were taken: a source file
    it is built from, or its launch configuration (the tuning in use)."""
    p = os.path.join(ROOT, "profiles", f"{name}.traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("src_hash") != source_hash(d["files"]) or d.get("tune") != tune:
            return None
    except (OSError, ValueError, KeyError):
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------- own arm

def run_own(args, dist):
    import torch
    import workload_inputs as inputs
    from collective_datapath_reduce_gb300 import _build
    from collective_datapath_reduce_gb300 import purlin as P

    _build.build()
    P.load()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.Stream(device=dev)
    wl = workloads(P, inputs, args.w4_mib)[args.workload]
    headline = args.workload == "allreduce_bf16_8x64MiB"
    if args.tune:
        wl.tune = dict(wl.tune or {}, **{k: int(v) for k, v in (f.split("=") for f in args.tune.split(","))})

    x = wl.make_inputs()                                      # host arrays, one per rank
    host_in = [torch.from_numpy(np.ascontiguousarray(a).view(np.uint8)).pin_memory() for a in x]
    src = [torch.empty(max(t.numel(), 1), dtype=torch.uint8, device=dev) for t in host_in]
    dst = [torch.empty(max(b, 1), dtype=torch.uint8, device=dev) for b in wl.out_bytes]
    with torch.cuda.stream(stream):
        for r in range(WORLD):
            if host_in[r].numel():
                src[r][:host_in[r].numel()].copy_(host_in[r], non_blocking=True)
    stream.synchronize()

    st, h = P.purlin_initialize(WORLD, None, 0, stream)
    P.check(st, "purlin_initialize")
    sptr = [t.data_ptr() for t in src]
    dptr = [t.data_ptr() for t in dst]

    def step():
        st = wl.call(h, sptr, dptr, stream)
        if st != P.PL_OK:
            raise P.PurlinError(st, wl.name)

    if wl.tune:
        P.check(P.purlin_tune_override(h, wl.tune), "purlin_tune_override")
    _, tune = P.purlin_tune_get(h, wl.coll, {"bf16": P.PL_BF16, "f32": P.PL_F32, "u8": P.PL_U8}[wl.dtype],
                                wl.tune_bytes)
    # The clock sampler starts first; the warm-up steps then run straight into
    # the timed region, so the GPU does not sit idle (and clock down) in between.
    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    stream.synchronize()
    K = args.steps
    dist.barrier()
    torch.cuda.synchronize(dev)
    # The timed region holds nothing but the K launches, back to back on the
    # launching stream (an event recorded between two launches would hold the
    # next one until the previous grid has fully retired), so the kernel's
    # average launch duration is the region's time over K.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    kernel_ms = total_ms / K
    time.sleep(0.1)
    clk = clocks.stop()
    st, dev_status = P.purlin_status_get(h, stream)
    P.check(st, "purlin_status_get")
    if dev_status:
        raise P.PurlinError(dev_status, "device")

    total_ms = dist.max(total_ms, dev)
    ms_per_step = total_ms / K
    value = dist.world * wl.algo_bytes * K / (total_ms / 1e3) / 1e9

    e2e = None
    if not args.device_only:
        # End to end: every step copies its inputs in from pinned host memory, runs
        # the collective and copies its outputs back.  Steps are pipelined over three
        # streams and two device buffer sets, so the host->device copy of step k+1
        # and the device->host copy of step k-1 overlap the kernel of step k.
        host_out = [torch.empty(b, dtype=torch.uint8).pin_memory() for b in wl.out_bytes]
        in_bytes = sum(t.numel() for t in host_in)
        out_bytes = sum(wl.out_bytes)
        Ke = K                                           # as many steps as the device-timed region
        src2 = [torch.empty_like(t) for t in src]
        dst2 = [torch.empty_like(t) for t in dst]
        sets = [([t.data_ptr() for t in src], [t.data_ptr() for t in dst], src, dst),
                ([t.data_ptr() for t in src2], [t.data_ptr() for t in dst2], src2, dst2)]
        # Each direction's per-rank copies are spread over NC streams, so several
        # copy engines work at once.
        NC = 4
        s_in = [torch.cuda.Stream(device=dev) for _ in range(NC)]
        s_out = [torch.cuda.Stream(device=dev) for _ in range(NC)]
        ev_in = [[torch.cuda.Event() for _ in range(NC)] for _ in range(Ke)]
        ev_done = [torch.cuda.Event() for _ in range(Ke)]
        ev_out = [[torch.cuda.Event() for _ in range(NC)] for _ in range(Ke)]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for q in s_in + s_out:
            q.wait_stream(stream)
        for k in range(Ke):
            sp, dp, sb, db = sets[k % 2]
            for c, q in enumerate(s_in):
                with torch.cuda.stream(q):
                    if k >= 2:
                        q.wait_event(ev_done[k - 2])      # step k-2 has finished reading this input set
                    for r in range(c, WORLD, NC):
                        if host_in[r].numel():
                            sb[r][:host_in[r].numel()].copy_(host_in[r], non_blocking=True)
                    ev_in[k][c].record(q)
            for c in range(NC):
                stream.wait_event(ev_in[k][c])
                if k >= 2:
                    stream.wait_event(ev_out[k - 2][c])   # step k-2's outputs have reached the host
            st = wl.call(h, sp, dp, stream)
            if st != P.PL_OK:
                raise P.PurlinError(st, wl.name)
            ev_done[k].record(stream)
            for c, q in enumerate(s_out):
                with torch.cuda.stream(q):
                    q.wait_event(ev_done[k])
                    for r in range(c, WORLD, NC):
                        if wl.out_bytes[r]:
                            host_out[r].copy_(db[r][:wl.out_bytes[r]], non_blocking=True)
                    ev_out[k][c].record(q)
        for q in s_in + s_out:
            stream.wait_stream(q)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
        e2e_ms = dist.max(e0.elapsed_time(e1), dev) / Ke
        staged = {"value": round(dist.world * wl.algo_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                  "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes, "ms_per_step": round(e2e_ms, 4),
                  "steps": Ke, "method": "staged: copy-engine copies in and out, h2d(k+1) and d2h(k-1) overlap the "
                  "kernel of step k; 4 copy streams per direction, 2 buffer sets"}
        del src2, dst2

        # End to end in place: the call is given the pinned host buffers themselves
        # and its kernel reads the inputs from host memory and writes the outputs
        # to host memory over the host link (the same bytes cross it each step).
        hp_in = [t.data_ptr() if t.numel() else None for t in host_in]
        hp_out = [t.data_ptr() if t.numel() else None for t in host_out]
        P.check(wl.call(h, hp_in, hp_out, stream), wl.name)   # builds the host-memory plan
        stream.synchronize()
        z0 = torch.cuda.Event(enable_timing=True)
        z1 = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize(dev)
        z0.record(stream)
        for _ in range(Ke):
            P.check(wl.call(h, hp_in, hp_out, stream), wl.name)
        z1.record(stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
        zc_ms = dist.max(z0.elapsed_time(z1), dev) / Ke
        e2e = {"value": round(dist.world * wl.algo_bytes / (zc_ms / 1e3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes, "ms_per_step": round(zc_ms, 4),
               "steps": Ke, "method": "in place: the C-ABI call takes the pinned host buffers, its kernel reads the "
               "inputs from host memory and writes the results to host memory", "staged": staged}

    peak, peak_kind = measured_peaks()
    achieved = wl.algo_bytes / (kernel_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(wl.name, tune),
                "peak_source": f"hbm_gbs of {peak_kind}", "kernel_ms": round(kernel_ms, 5),
                "kernel_ms_source": "timed region / K: nothing but back-to-back launches of the kernel on its stream",
                "algorithmic_bytes_per_launch": wl.algo_bytes}

    extras = None
    if headline and not args.no_extras and dist.rank == 0:
        extras = side_table(P, h, stream, dev)

    P.check(P.purlin_finalize(h, stream), "purlin_finalize")

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl, x, budget_s=12.0)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": config_of(wl, x),
        "parallelism": f"replicas{dist.world}" if dist.world > 1 else "single-gpu",
        "tune": tune,
        "roofline": roofline, "e2e": e2e, "gpu_launches": K, "clocks": clk,
        "cpu_baseline": cpu,
        "pct_of_hbm_peak": round(100 * value / dist.world / peak, 2),
    }
    if extras:
        line["vs_size"] = extras
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def side_table(P, h, stream, dev):
    """The metric against size: GB/s (algorithmic bytes) and microseconds per
    call for every collective over the workloads' size range, the two-shot
    AllReduce layout, the two Atoms, and the device-to-device copy of the same
    traffic.  Each library point is a CUDA graph of 10 calls (the pages'
    graphLaunches knob): 5 warm-up replays, then 20 timed replays, each after
    a write of twice the L2 size; the point gives the median and the 10th /
    90th percentiles of the time per call.  Points whose working set fits in
    the L2 are marked: after the first call of a replay they run from the L2.
    Collective points also give the pages' own figure, totalBytes over time
    (input bytes per rank; the output size for AllGather).  The copy
    reference is 10 plain launches of torch's copy kernel."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    GRAPH, WARM, RUNS = 10, 5, 20
    MI = 1 << 20
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * MI))
    peak, _ = measured_peaks()
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def timeit(fn, graph=True):
        """Per-call milliseconds of each timed run."""
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            stream.synchronize()
            g = None
            if graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(GRAPH):
                        fn()
            def run():
                if g is not None:
                    g.replay()
                else:
                    for _ in range(GRAPH):
                        fn()
            for _ in range(WARM):
                run()
            times = []
            for k in range(RUNS):
                flush.fill_(k & 0xFF)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                run()
                b.record(stream)
                stream.synchronize()
                times.append(a.elapsed_time(b) / GRAPH)
            del g
            return times

    def bufs(n, count, dtype=torch.uint8):
        if dtype == torch.uint8:
            return [torch.randint(0, 256, (max(n, 1),), dtype=torch.uint8, device=dev, generator=gen)
                    for _ in range(count)]
        return [torch.randn(max(n, 1), dtype=dtype, device=dev, generator=gen) for _ in range(count)]

    def point(nbytes, times, total_bytes=None):
        # the algorithmic bytes are the distinct bytes a call touches: its working set.
        # total_bytes: the pages' own bandwidth convention (purlin bench: input bytes
        # per rank, the output size for AllGather), reported beside it for context.
        t = sorted(times)
        med = statistics.median(t)
        pct = lambda q: t[min(len(t) - 1, int(q * (len(t) - 1) + 0.5))]
        d = {"bytes": nbytes, "us": round(med * 1e3, 2), "us_p10": round(pct(0.1) * 1e3, 2),
             "us_p90": round(pct(0.9) * 1e3, 2), "GB/s": round(nbytes / (med / 1e3) / 1e9, 1),
             "pct_of_peak": round(100 * nbytes / (med / 1e3) / 1e9 / peak, 1)}
        if total_bytes is not None:
            d["totalBytes_GB/s"] = round(total_bytes / (med / 1e3) / 1e9, 1)
        if nbytes <= l2:
            d["l2_resident"] = True
        return d

    out = {"d2d_copy": {}, "launch_floor": {}, "all_gather_u8": {}, "all_to_all_u8": {}, "all_reduce_bf16": {},
           "reduce_scatter_f32": {}, "all_reduce_two_shot_bf16": {}, "all_reduce_two_shot_fused_bf16": {},
           "all_reduce_ring_bf16": {},
           "reduce_scatter_v_bf16": {},
           "device_api_fused": {}, "atom_copy": {}, "atom_reduce": {}}
    chk = lambda st: P.check(st)
    for size in [1 << (10 + 2 * k) for k in range(10)]:          # 1 KiB .. 256 MiB per rank
        key = f"{size >> 10}KiB" if size < MI else f"{size >> 20}MiB"
        src = bufs(size, WORLD)
        dag = [torch.empty(WORLD * size, dtype=torch.uint8, device=dev) for _ in range(WORLD)]
        out["all_gather_u8"][key] = point(WORLD * size * (1 + WORLD),
                                          timeit(lambda: chk(P.purlin_all_gather(h, src, dag, size, stream))),
                                          WORLD * size)
        del dag
        da = [torch.empty(size, dtype=torch.uint8, device=dev) for _ in range(WORLD)]
        out["all_to_all_u8"][key] = point(2 * WORLD * size,
                                          timeit(lambda: chk(P.purlin_all_to_all(h, src, da, size, stream))), size)
        big = torch.empty(2 * WORLD * size, dtype=torch.uint8, device=dev)
        half = WORLD * size
        # the copy kernel torch launches outside a graph (inside one, copy_ becomes
        # a copy-engine memcpy node, which is slower than an SM copy)
        out["d2d_copy"][key] = point(2 * half, timeit(lambda: big[half:].copy_(big[:half]), graph=False))
        del src, da, big
        torch.cuda.empty_cache()
    # the floor of a call in a CUDA graph of 10: torch's one-element fill kernel
    tiny = torch.zeros(1, dtype=torch.float32, device=dev)
    out["launch_floor"] = {"torch_fill_1_element": point(4, timeit(lambda: tiny.fill_(1.0)))}
    for size in (64 << 10, 1 * MI, 16 * MI, 64 * MI, 256 * MI):
        key = f"{size >> 10}KiB" if size < MI else f"{size >> 20}MiB"
        x = bufs(size // 2, WORLD, torch.bfloat16)
        y = [torch.empty_like(t) for t in x]
        out["all_reduce_bf16"][key] = point(2 * WORLD * size, timeit(
            lambda: chk(P.purlin_all_reduce(h, x, y, size, P.PL_BF16, 0, stream))), size)
        if size >= 16 * MI:
            one_shot = [t.clone() for t in y]
            for layout, name in ((P.PL_LAYOUT_TWO_SHOT, "all_reduce_two_shot_bf16"),
                                 (P.PL_LAYOUT_TWO_SHOT_FUSED, "all_reduce_two_shot_fused_bf16"),
                                 (P.PL_LAYOUT_RING, "all_reduce_ring_bf16")):
                P.check(P.purlin_tune_override(h, {"layout": layout}))
                for t in y:
                    t.fill_(float("nan"))
                out[name][key] = point(2 * WORLD * size, timeit(
                    lambda: chk(P.purlin_all_reduce(h, x, y, size, P.PL_BF16, 0, stream))), size)
                out[name][key]["max_ulp_vs_one_shot"] = max_ulp_dev(y, one_shot, stream)
            P.check(P.purlin_tune_override(h, None))
            del one_shot
        del x, y
        x = bufs(size // 4, WORLD, torch.float32)
        y = [torch.empty(size // 4 // WORLD, dtype=torch.float32, device=dev) for _ in range(WORLD)]
        out["reduce_scatter_f32"][key] = point(WORLD * size + size, timeit(
            lambda: chk(P.purlin_reduce_scatter(h, x, y, size, P.PL_F32, 0, stream))), size)
        del x, y
        torch.cuda.empty_cache()
    # the allocation-free AllReduce entry point (two-shot, scratch in a static
    # device array; no handle), timed in plain launches
    out["all_reduce_noalloc_bf16"] = {}
    dstat = torch.zeros(1, dtype=torch.int32, device=dev)
    for size in (16 * MI, 64 * MI, 256 * MI):
        x = bufs(size // 2, WORLD, torch.bfloat16)
        y = [torch.empty_like(t) for t in x]
        one_shot = [torch.empty_like(t) for t in x]
        chk(P.purlin_all_reduce(h, x, one_shot, size, P.PL_BF16, 0, stream))
        key = f"{size >> 20}MiB"
        out["all_reduce_noalloc_bf16"][key] = point(2 * WORLD * size, timeit(
            lambda: chk(P.purlin_all_reduce_noalloc(WORLD, x, y, size, P.PL_BF16, dstat, stream)), graph=False), size)
        if int(dstat.item()) != 0:
            raise RuntimeError("allocation-free AllReduce reported a device error")
        out["all_reduce_noalloc_bf16"][key]["max_ulp_vs_one_shot"] = max_ulp_dev(y, one_shot, stream)
        del x, y, one_shot
    torch.cuda.empty_cache()
    # ReduceScatterV: uneven chunks (workload 5's first row of counts), bf16
    import workload_inputs as _inputs
    C5, _ = _inputs.w5_counts(WORLD)
    counts = [int(v) * 2 for v in C5[0]]
    total = sum(counts)
    x = bufs(total // 2, WORLD, torch.bfloat16)
    y = [torch.empty(max(c, 2) // 2, dtype=torch.bfloat16, device=dev) for c in counts]
    out["reduce_scatter_v_bf16"][f"{total >> 20}MiB"] = point(WORLD * total + total, timeit(
        lambda: chk(P.purlin_reduce_scatter_v(h, x, y, counts, P.PL_BF16, 0, stream))))
    del x, y
    # Device-side API: the example kernel calling purlin::all_gather /
    # all_reduce with no work of its own, one cooperative launch per call
    from collective_datapath_reduce_gb300 import examples as EX
    size = 64 * MI
    for which, nm, nb_in, nb_out, alg in ((EX.AG, "all_gather_u8_8x64MiB", size, WORLD * size, 9 * WORLD * size),
                                          (EX.AR_BF16, "all_reduce_bf16_8x64MiB", size, size, 2 * WORLD * size)):
        src = bufs(nb_in, WORLD)
        dst = [torch.empty(nb_out, dtype=torch.uint8, device=dev) for _ in range(WORLD)]
        bar = torch.zeros(2, dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        f = EX.FusedArgs()
        f.ctx.world = WORLD
        for r in range(WORLD):
            f.ctx.src[r] = src[r].data_ptr()
            f.ctx.dst[r] = dst[r].data_ptr()
        f.ctx.barrier = bar.data_ptr()
        f.bytes, f.out_bytes, f.which, f.work = nb_in, nb_out, which, 0
        # the grid is the caller's choice: one CTA per SM for the AllGather
        # (measured best), every resident CTA for the AllReduce
        g = EX.max_grid()
        if which == EX.AG:
            g = min(g, torch.cuda.get_device_properties(dev).multi_processor_count)
        f.coll_blocks = g
        f.status = status.data_ptr()
        times = timeit(lambda: EX.launch(f, g, stream.cuda_stream), graph=False)
        if int(status.item()) != 0:
            raise RuntimeError("device-side collective reported a time-out")
        out["device_api_fused"][nm] = point(alg, times)
        del src, dst
    torch.cuda.empty_cache()
    for size in (64 * MI, 256 * MI):
        a = bufs(size, 1)[0]
        b = torch.empty(size, dtype=torch.uint8, device=dev)
        out["atom_copy"][f"1to1_{size >> 20}MiB"] = point(2 * size, timeit(
            lambda: chk(P.purlin_atom_copy(h, a, [b], size, stream))))
        del a, b
    size = 64 * MI
    for dt, code, nm in ((torch.bfloat16, P.PL_BF16, "bf16"), (torch.float32, P.PL_F32, "f32")):
        x = bufs(size // (2 if nm == "bf16" else 4), WORLD, dt)
        for nd in (1, WORLD):
            y = [torch.empty_like(x[0]) for _ in range(nd)]
            out["atom_reduce"][f"{nm}_8to{nd}_64MiB"] = point((WORLD + nd) * size, timeit(
                lambda: chk(P.purlin_atom_reduce(h, x, y, size, code, stream))))
            del y
        del x
    torch.cuda.empty_cache()
    return out


def max_ulp_dev(got, want, stream):
    """Largest ulp distance between two lists of bf16 tensors, on the device:
    bit patterns folded to ordered integers (negative values to minus their
    magnitude bits), then the largest difference.  0 = bit-identical."""
    import torch
    m = 0
    with torch.cuda.stream(stream):
        for g, w in zip(got, want):
            a = g.view(torch.int16).to(torch.int32)
            b = w.view(torch.int16).to(torch.int32)
            a = torch.where(a < 0, -(a & 0x7FFF), a)
            b = torch.where(b < 0, -(b & 0x7FFF), b)
            m = max(m, int((a - b).abs().max().item()))
    return m


# ---------------------------------------------------------- CPU baseline

def config_of(wl, x):
    """The workload a line measures (identical in both arms): what it is, its
    size, and how its working set compares with the GPU's L2."""
    in_bytes = sum(int(np.asarray(a).nbytes) for a in x)
    out_bytes = sum(wl.out_bytes)
    return {"workload": wl.desc, "name": wl.name, "world": WORLD, "algorithmic_bytes_per_step": wl.algo_bytes,
            "l2": f"inputs {in_bytes >> 20} MiB and outputs {out_bytes >> 20} MiB per step exceed the 126 MiB "
                  "L2; no flush between steps"}


def host_cpu():
    """Core count and CPU model of this host (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu model")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.machine()}


def _reference_call(name):
    """The oracle function of a workload: f(list of rank arrays) -> outputs."""
    import oracle
    import workload_inputs as inputs
    C5, c5 = inputs.w5_counts(WORLD)
    return {
        "allreduce_bf16_8x64MiB": lambda ins: oracle.all_reduce(ins, "bf16"),
        "allreduce_two_shot_bf16_8x64MiB": lambda ins: oracle.all_reduce(ins, "bf16"),
        "allreduce_ring_bf16_8x64MiB": lambda ins: oracle.all_reduce(ins, "bf16"),
        "reduce_scatter_f32_8x256MiB": lambda ins: oracle.reduce_scatter(ins, "f32"),
        "reduce_scatter_bf16_8x128MiB": lambda ins: oracle.reduce_scatter(ins, "bf16"),
        "all_gather_u8_8x256MiB": oracle.all_gather,
        "all_to_all_u8_8x256MiB": oracle.all_to_all,
        "all_to_all_v_bf16_w5": lambda ins: oracle.all_to_all_v(ins, C5),
        "all_gather_v_bf16_w5": lambda ins: oracle.all_gather_v(ins, [int(v) for v in c5]),
    }[name]


class OracleRun:
    """The workload's oracle, as it stands, on a bounded sample: the first
    `k` elements of every rank (whole chunks for ReduceScatter / AllToAll), or
    the whole workload for the V collectives, whose counts fix the layout.
    A run's throughput counts the sample's share of the algorithmic bytes."""

    def __init__(self, wl, x, run_budget_s):
        self.fn = _reference_call(wl.name)
        self.x = [np.asarray(a) for a in x]
        self.algo_bytes = wl.algo_bytes
        if wl.name.endswith("_w5"):
            self.k, self.frac = None, 1.0
        else:
            n = self.x[0].size
            probe = min(n, 1 << 20)
            probe -= probe % (8 * WORLD)
            t = self.run_once(probe)
            k = int(min(n, max(1 << 16, probe * run_budget_s / max(t, 1e-4))))
            self.k = k - k % (8 * WORLD)
            self.frac = self.k / n

    def run_once(self, k=None):
        k = self.k if k is None else k
        ins = self.x if k is None else [a[:k] for a in self.x]
        t0 = time.perf_counter()
        self.fn(ins)
        return time.perf_counter() - t0

    def gbs(self, seconds):
        return self.algo_bytes * self.frac / seconds / 1e9

    def sample(self):
        what = ("the whole workload per run" if self.k is None else
                f"first {self.k} of {self.x[0].size} elements of each of the {WORLD} ranks per run")
        return what + " (numpy, single-threaded)"


def cpu_baseline(wl, x, budget_s=12.0):
    """The CPU oracle of the workload, as it stands, for about budget_s seconds."""
    o = OracleRun(wl, x, run_budget_s=budget_s / 8)
    reps, spent = 0, 0.0
    while spent < budget_s and reps < 50:
        spent += o.run_once()
        reps += 1
    per = spent / reps
    return dict({"value": round(o.gbs(per), 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                 "sample": f"{o.sample()}, {reps} runs, {per:.3f} s each",
                 "sampled_fraction": round(o.frac, 6)}, **host_cpu())


# ----------------------------------------------------------- reference arm

def run_reference(args, dist):
    """The oracle of the selected workload times itself on the host cores, on
    a bounded sample (the first elements of every rank; the V workloads in
    full); rank 0 only."""
    if dist.rank != 0:
        return
    import workload_inputs as inputs
    from collective_datapath_reduce_gb300 import purlin as P  # names only: the library is not loaded
    wl = workloads(P, inputs)[args.workload]
    x = [np.asarray(a) for a in wl.make_inputs()]
    steps = args.steps + args.warmup
    o = OracleRun(wl, x, run_budget_s=max(0.05, 120.0 / max(steps, 1)))
    for _ in range(args.warmup):
        o.run_once()
    times = [o.run_once() for _ in range(args.steps)]
    per = sum(times) / len(times)
    value = round(o.gbs(per), 4)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": config_of(wl, x),
        "sampled_fraction": round(o.frac, 6), "input_elements": sum(a.size for a in x),
        "cpu_baseline": dict({"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                              "sample": o.sample()}, **host_cpu()),
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main():
    args = parse()
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
        return
    run_own(args, dist)


if __name__ == "__main__":
    main()
