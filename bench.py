"""Throughput of the GB300 gate-level re-simulator on the 1M-gate workload.

A step is one re-simulation of the whole netlist (all 40 logic levels, every gate in
every one of the 256 cycle windows: Algorithm 1, the output-offset scan, the stores
and the TC/T1 reduction) with the input waveforms already resident in HBM.

Prints one JSON line (rank 0):
  value      output toggle events per second over device time (sum of TC / time)
  e2e        the same metric through the C ABI with host buffers, every step: H2D of
             the whole-testbench input waveforms, their cut into cycle windows on the
             GPU, simulate, D2H of the toggle statistics (and, for comparison, the same
             with windows cut on the host beforehand)
  roofline   the level kernel against the measured HBM copy bandwidth, on
             algorithmic bytes (each consumed waveform read once per run, each
             output written once, 8 B of window index per consumed (net, window)
             and per (gate, window), descriptors once)
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

``--impl reference`` times the CPU oracle instead (a plain event-driven simulator,
windows spread over the host cores), on a bounded sample per step.
Under torchrun (N ranks, one GPU each) the windows are split over the GPUs: the
testbench is N times longer, rank r simulates the r-th contiguous range of its
windows (as many as one GPU does alone: weak scaling), and the per-gate TC/T1 are
summed over the ranks once; rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "output toggle events/sec and gate-cycles/sec at 1 GB300; % of HBM roofline"
UNIT = "output toggle events/s"
WORKLOAD = "1M"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ("gate_level_logic_gb300/csrc/lane.cuh", "gate_level_logic_gb300/csrc/level_kernel.cu",
                  "gate_level_logic_gb300/csrc/gatspi_internal.cuh")


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _init_pg(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


WORKLOAD_NAMES = {
    "1M": ("1M-gate synthetic netlist, 40 levels, 9-cell mix with SDF-conditional arcs; "
           "4096 inputs, 10k cycles x period 1000, 5% activity, 10% glitch pairs; 256 cycle windows"),
    "5M": ("5M-gate synthetic netlist, 60 levels, 9-cell mix, 30% of multi-input cells with SDF-conditional "
           "arcs; 16384 inputs, 2000 cycles x period 1000, 20% activity; 128 cycle windows"),
    "scan500k": ("500k-gate scan-style netlist of NAND2/NOR2/XOR2, 30 levels; 4096 inputs, 100k cycles x "
                 "period 1000, 2% activity; 256 cycle windows"),
}


def workload_config(net, stim, pulse_percent=100, overrides=None, workload=WORKLOAD, world=1, compact=False):
    name = WORKLOAD_NAMES[workload]
    if world > 1:
        name += ("; the testbench %dx longer, its windows split into %d contiguous ranges, one per GPU"
                 % (world, world))
    extra = {}
    if overrides:
        name = "not the default workload: " + name + ", with the overrides listed"
        extra["overrides"] = overrides
    return {
        "workload": name,
        "gates": int(net.num_gates), "levels": int(net.num_levels), "inputs": int(net.num_inputs),
        "edges": int(net.num_edges), "windows": int(stim.num_windows), "cycles": int(stim.window_cycles.sum()),
        "pulse_percent": pulse_percent,
        "packed_levels": bool(compact),
        "parallelism": ("windows split over %d GPUs (one contiguous range each, one int64 sum of TC/T1 "
                        "at the end)" % world) if world > 1 else "one GPU",
        "l2": "inputs larger than L2 (waveform pool of several GB per step, no flush needed)",
        **extra,
    }


def algorithmic_bytes(net, net_words, W):
    """Algorithmic bytes of one run (every level): each consumed (net, window) waveform
    read once, each output written once, 8 B of window index per consumed (net,
    window) and per (gate, window), and the gate descriptors once (16 B per gate and
    per fanin edge).  ``net_words``: words of every net over all its windows.
    Returns (total, parts)."""
    P, G = net.num_inputs, net.num_gates
    net_words = np.asarray(net_words, np.int64)
    consumed = np.unique(net.fanin_net)
    parts = {
        "read_waveforms": 4 * int(net_words[consumed].sum()),
        "write_waveforms": 4 * int(net_words[P:].sum()),
        "window_index": 8 * W * (int(consumed.size) + G),
        "descriptors": 16 * G + 16 * int(net.num_edges),
    }
    return sum(parts.values()), parts


def demand_bytes(net, net_words, W):
    """Per level: the waveforms of every distinct source net of the level read (a net
    consumed by several levels counts in each), the level's outputs written, their
    window index read and written, and the level's gate descriptors."""
    P = net.num_inputs
    net_words = np.asarray(net_words, np.int64)
    lo = net.level_offsets
    out = []
    for lvl in range(net.num_levels):
        g0, g1 = int(lo[lvl]), int(lo[lvl + 1])
        srcs = np.unique(net.fanin_net[net.fanin_off[g0]:net.fanin_off[g1]])
        read = 4 * int(net_words[srcs].sum()) + 8 * W * srcs.size
        write = 4 * int(net_words[P + g0:P + g1].sum()) + 8 * W * (g1 - g0)
        desc = 16 * (g1 - g0) + 16 * int(net.fanin_off[g1] - net.fanin_off[g0])
        out.append(read + write + desc)
    return np.array(out, dtype=np.int64)


def _code_only(text):
    """Source text without // comments and blank lines: a comment edit leaves the
    compiled kernel, and so its measured counters, unchanged."""
    lines = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            lines.append(code)
    return "\n".join(lines)


def _kernel_hash(read=None):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(_code_only(text).encode())
    return h.hexdigest()[:16]


# The plan ranks a gate's windows by bound up to this many windows per context and
# takes more in window order (the window index's perm is unused beyond it).
RANKED_WINDOWS = 1024

# How a run's levels are simulated, which decides the kernel its roofline describes
# and the ncu record its DRAM traffic is scaled from (None: no record).
SIM_REGIMES = {
    "ranked": ("level_kernel (one launch per logic level; windows ranked by bound)",
               "level_kernel_small_traffic.json"),
    "window_order": ("level_kernel (one launch per logic level; windows in window order)",
                     "level_kernel_4096windows_traffic.json"),
    "cut": ("level_order_kernel + level_chunk_kernel (one pair per logic level; windows cut into time chunks)",
            None),
}


def sim_regime(lanes_per_window, windows):
    """The regime of a context with `windows` windows whose windows get
    `lanes_per_window` lanes each (more than one: cut into time chunks)."""
    if lanes_per_window > 1:
        return "cut"
    return "ranked" if windows <= RANKED_WINDOWS else "window_order"


def _traffic(demand_per_launch, regime, pulse_percent=100):
    """DRAM bytes per simulation launch: the ratio of DRAM traffic to demand bytes that
    ncu measured on the committed small case of the same regime (the same kernel
    source, PATHPULSEPERCENT = 100, two launches), applied to this workload's mean
    demand bytes per launch.  (None, None, None) when the regime has no record, the
    run uses another PATHPULSEPERCENT (another instantiation of the kernel), or the
    record is missing or was taken on other kernel code."""
    name = SIM_REGIMES[regime][1]
    if name is None or pulse_percent != 100:
        return None, None, None
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, None, None
    if rec.get("kernel_sha") != _kernel_hash():
        return None, None, None
    ratio = float(rec["dram_bytes"]) / float(rec["demand_bytes"])
    return ratio * float(demand_per_launch), ratio, name


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = list(csv.reader(io.StringIO(getattr(self, "out", "") or "")))
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(net, stim, seconds_target=15.0, pulse_percent=100):
    """The CPU oracle as it stands, windows spread over all host cores, on a bounded
    sample of the workload's windows (all gates)."""
    import oracle
    cores = os.cpu_count() or 1
    W = stim.num_windows
    n = max(1, min(W, cores))
    sel = np.linspace(0, W - 1, n).astype(np.int64)
    t = time.perf_counter()
    r = oracle.simulate(net, synth_select(stim, sel), threads=cores, pulse_percent=pulse_percent)
    dt = time.perf_counter() - t
    # grow the sample once to land near the target duration
    if dt < seconds_target / 4 and n < W:
        n2 = int(min(W, max(n + 1, n * min(8.0, seconds_target / max(dt, 1e-3)))))
        sel = np.linspace(0, W - 1, n2).astype(np.int64)
        t = time.perf_counter()
        r = oracle.simulate(net, synth_select(stim, sel), threads=cores, pulse_percent=pulse_percent)
        dt = time.perf_counter() - t
    events = int(r.tc.sum())
    cycles = int(stim.window_cycles[sel].sum())
    return {
        "value": events / dt, "unit": UNIT, "cores": min(cores, len(sel)), "kind": "oracle",
        "sample": "%d of %d windows (all %d gates, %d cycles), %.1f s" % (len(sel), W, net.num_gates, cycles, dt),
        "gate_cycles_per_s": net.num_gates * cycles / dt,
    }


def synth_select(stim, sel):
    import synth
    return synth.select_windows(stim, sel)


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    import synth
    import oracle
    oracle.build()
    workload = getattr(args, "workload", WORKLOAD)
    net, stim = synth.make(workload)
    cores = os.cpu_count() or 1
    W = stim.num_windows
    n = min(W, 2 * cores)
    sel = np.linspace(0, W - 1, n).astype(np.int64)
    sub = synth.select_windows(stim, sel)
    for _ in range(args.warmup):
        oracle.simulate(net, sub, threads=cores, pulse_percent=args.pulse_percent)
    times, events = [], 0
    for _ in range(args.steps):
        t = time.perf_counter()
        r = oracle.simulate(net, sub, threads=cores, pulse_percent=args.pulse_percent)
        times.append(time.perf_counter() - t)
        events += int(r.tc.sum())
    total = sum(times)
    value = events / total
    cycles = int(stim.window_cycles[sel].sum())
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": workload_config(net, stim, args.pulse_percent, workload=workload),
        "gate_cycles_per_s": net.num_gates * cycles * args.steps / total,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, n), "kind": "oracle",
                         "sample": "%d of %d windows per step (all gates)" % (n, W)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def _e2e(args, sim, inputs, net, stream, dist, events_per_step, testbench):
    """Same metric through the public API with host buffers: every step copies the
    inputs in (and, with ``testbench``, cuts the whole-testbench waveforms into windows
    on the GPU), simulates and reads the statistics back; with several ranks, each
    rank's statistics are then summed over the ranks (the run's one collective)."""
    import torch
    from gate_level_logic_gb300 import shard
    pin_off = torch.from_numpy(np.ascontiguousarray(inputs[0], np.int64)).pin_memory()
    pin_words = torch.from_numpy(np.ascontiguousarray(inputs[1], np.int32)).pin_memory()
    load = sim.load_testbench if testbench else sim.load
    e2e_steps = max(1, args.steps)
    _barrier(dist)
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(e2e_steps):
        load(pin_off, pin_words, stream=stream)
        sim.simulate(stream=stream)
        tc_e, t1_e, _ = sim.toggle_stats_view()   # the statistics in host memory, no extra copy
        if dist is not None:
            local = int(tc_e.sum())
            tc_e, t1_e = shard.sum_stats(dist, tc_e.astype(np.int64), t1_e.astype(np.int64))
    torch.cuda.synchronize()
    e2e_s = _max_over_ranks(dist, time.perf_counter() - t)
    assert (local if dist is not None else int(tc_e.sum())) == events_per_step
    e2e_value = _sum_over_ranks(dist, events_per_step * e2e_steps) / e2e_s
    h2d = pin_off.numel() * 8 + pin_words.numel() * 4
    d2h = 2 * 8 * net.num_gates + 16       # TC and T1 per gate, status word

    return e2e_value, h2d, d2h


def _testbench_cut(args, sim, tb, stream, with_oracle):
    """Time the device-side cut of the whole-testbench waveforms into windows
    (gatspi_load_testbench from device memory: format check + cut + window index),
    and, for scale, the oracle's host cut of the same testbench on one core."""
    import torch
    d_off = torch.from_numpy(np.ascontiguousarray(tb.off, np.int64)).cuda()
    d_words = torch.from_numpy(np.ascontiguousarray(tb.words, np.int32)).cuda()
    for _ in range(3):
        sim.load_testbench(d_off, d_words, stream=stream)
    reps = 20
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(reps):
        sim.load_testbench(d_off, d_words, stream=stream)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / reps
    out = {"gpu_ms": ms, "testbench_words": int(tb.words.size), "note": "per call, host synchronisation included"}
    if with_oracle:
        import oracle
        oracle.build()
        t = time.perf_counter()
        _, words = oracle.restructure(tb.off, tb.words, tb.window_len)
        out["oracle_cpu_ms"] = 1e3 * (time.perf_counter() - t)
        out["window_words"] = int(words.size)
    return out


def _sdf_translate(with_oracle):
    """SDF text -> delay tables: the library's translator (host code) against the
    oracle's translation of the same text, in MB of SDF per second."""
    import synth
    from gate_level_logic_gb300 import sdf_annotate
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=4000, num_inputs=128, num_levels=12, seed=1,
                                                   cond_cells=("AOI21", "MUX2", "OAI22", "NAND4"),
                                                   cond_fraction=0.5))
    s = synth.write_sdf(net, seed=1, file_unit="1ns")
    args = (s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names, net.fanin_off, net.gate_dly_off,
            net.dly_data.size, 1000)
    mb = len(s.text) / 1e6
    t = time.perf_counter()
    dly, _, _ = sdf_annotate(*args)
    lib_s = time.perf_counter() - t
    assert np.array_equal(dly, net.dly_data)
    out = {"sdf_mb": mb, "gates": net.num_gates, "library_mb_per_s": mb / lib_s}
    if with_oracle:
        from oracle import sdf as osdf
        t = time.perf_counter()
        osdf.annotate(*args)
        out["oracle_mb_per_s"] = mb / (time.perf_counter() - t)
    return out


def run_gpu(args):
    import torch

    import synth
    from gate_level_logic_gb300 import build, shard

    rank, world, local = _dist()
    dist = _init_pg(world)
    torch.cuda.set_device(local)
    build.build()
    over = {}
    if args.windows:
        over["windows"] = args.windows
    if args.cycles:
        over["cycles"] = args.cycles
    if args.gates:
        over["net_num_gates"] = args.gates
    workload = args.workload
    if args.sweep:
        activity, windows = args.sweep.split(":")
        net, stim = synth.sweep(float(activity), int(windows))
        over = {"sweep_point": {"activity": float(activity), "windows": int(windows), "stimulus_seed": 4,
                                "glitch_pairs": 0.0}}
    else:
        kw = dict(over)
        if world > 1:
            # weak scaling: every rank simulates as many windows as one GPU does alone,
            # its own contiguous range of one testbench that many times longer
            _, stim_kw = synth.WORKLOADS[workload]
            kw["cycles"] = world * int(kw.get("cycles", stim_kw["cycles"]))
            kw["windows"] = world * int(kw.get("windows", stim_kw["windows"]))
        net, stim = synth.make(workload, **kw)
    flags = (0x8 if args.compact else 0) | (0x10 if args.whole_windows else 0)   # COMPACT, WHOLE_WINDOWS
    pool_gb = args.pool_gb if args.pool_gb > 0 else {"1M": 48.0, "5M": 170.0, "scan500k": 64.0}[workload]
    pool_words = int(pool_gb * (1 << 30) / 4)
    part = shard.WindowShard(net, stim.window_len, world, rank, pool_words=pool_words, flags=flags,
                             pulse_percent=args.pulse_percent)
    sim = part.sim
    stream = torch.cuda.current_stream()
    part.load(stim.pi_off, stim.pi_words, stream=stream)
    lanes_per_window = sim.lanes_per_window()   # > 1: windows cut into time chunks
    rank_off, rank_words = shard.slice_windows(stim.pi_off, stim.pi_words, net.num_inputs, stim.num_windows,
                                               part.w0, part.w1)
    W = part.w1 - part.w0                           # this rank's windows

    for _ in range(max(args.warmup, 1)):
        sim.simulate(stream=stream)
    tc, t0, t1 = sim.toggle_stats()
    events_per_step = int(tc.sum())                 # this rank's
    _, net_words = sim.net_digests(with_words=True)
    run_bytes, run_parts = algorithmic_bytes(net, net_words, W)
    lvl_demand = demand_bytes(net, net_words, W)
    waveform_words = int(net_words.sum())
    if args.dump_levels and rank == 0:
        with open(args.dump_levels, "w") as f:
            json.dump({"demand_bytes": lvl_demand.tolist(), "algorithmic_bytes_per_run": run_bytes,
                       "algorithmic_parts": run_parts}, f)
    pool_used = sim.pool_used()

    # ---- timed region: device time, inputs resident ----------------------------
    # The step as a user runs it: the captured level graph, each kernel starting in
    # the previous one's tail.  Then the same steps again with CUDA events around
    # every kernel (which serialises them) for the per-kernel times of the roofline.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    level_ms = np.zeros(net.num_levels, np.float64)      # simulation kernel of every level
    bounds_ms = np.zeros(net.num_levels, np.float64)     # planning + placement kernels of every level
    serial_ms = []
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            starts[k].record(stream)
            sim.simulate(stream=stream)
            ends[k].record(stream)
        torch.cuda.synchronize()
        _barrier(dist)
        sim.set_level_timing(True)
        sim.simulate(stream=stream)                       # warm the direct launches
        sim.sync()
        for k in range(args.steps):
            t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0e.record(stream)
            sim.simulate(stream=stream)
            t1e.record(stream)
            sim.sync()
            serial_ms.append(t0e.elapsed_time(t1e))
            lt, bt = sim.level_times()
            level_ms += lt
            bounds_ms += bt
        sim.set_level_timing(False)
        torch.cuda.synchronize()
    _barrier(dist)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = _max_over_ranks(dist, sum(step_ms) / 1e3)
    all_events = _sum_over_ranks(dist, events_per_step * args.steps)
    value = all_events / total_s
    gate_cycles = net.num_gates * int(stim.window_cycles[part.w0:part.w1].sum())   # this rank's windows
    lo = np.asarray(net.level_offsets)
    launches_per_step = int(2 * net.num_levels + np.count_nonzero(np.diff(lo)))
    gate_cycles_per_s = _sum_over_ranks(dist, gate_cycles * args.steps) / total_s

    # roofline of the level kernel: the run's algorithmic bytes per launch (one launch
    # per level) over its mean launch time, i.e. all of them over its total time
    kern_s = level_ms.sum() / 1e3
    achieved = float(run_bytes * args.steps / kern_s / 1e9)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            peak = float(json.load(f)["hbm_gbs"])
        peak_src = "measured"
    else:
        peak, peak_src = 6800.0, "fallback"
    regime = sim_regime(lanes_per_window, W)
    traffic, traffic_ratio, traffic_rec = _traffic(float(lvl_demand.mean()), regime, args.pulse_percent)

    # ---- end to end through the C ABI: host buffers, copies inside the region ---
    if args.no_e2e or args.sweep:      # no end-to-end legs on sweep points
        e2e_value, h2d, d2h, e2e_win, cut = None, 0, 0, None, None
    elif world > 1:                    # each rank copies its own windows in
        e2e_win = _e2e(args, sim, (rank_off, rank_words), net, stream, dist, events_per_step, False)
        e2e_value, h2d, d2h, cut = e2e_win[0], e2e_win[1], e2e_win[2], None
    else:
        tb = synth.testbench(workload, **over)
        e2e_value, h2d, d2h = _e2e(args, sim, (tb.off, tb.words), net, stream, dist, events_per_step, True)
        e2e_win = _e2e(args, sim, (stim.pi_off, stim.pi_words), net, stream, dist, events_per_step, False)
        cut = _testbench_cut(args, sim, tb, stream, rank == 0 and not args.no_cpu_baseline)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": workload_config(net, stim, args.pulse_percent, over, workload, world, args.compact),
        "lanes_per_window": lanes_per_window,
        "gate_cycles_per_s": gate_cycles_per_s,
        "events_per_step": events_per_step,
        "pool_words_used": pool_used,
        "waveform_words": waveform_words,
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_source": peak_src,
            "kernel": SIM_REGIMES[regime][0],
            "algorithmic_bytes_per_launch": float(run_bytes) / net.num_levels,
            "algorithmic_bytes_per_step": run_parts,
            "demand_bytes_per_launch": float(lvl_demand.mean()),
            "traffic_note": None if traffic is None else
            "ncu DRAM bytes / demand bytes = %.3f on the committed small case "
            "(profiles/%s), times this workload's demand bytes per launch" % (traffic_ratio, traffic_rec),
            "step_achieved_gbs": float(run_bytes * args.steps / total_s / 1e9),
            "avg_launch_ms": float(level_ms.sum() / (args.steps * net.num_levels)),
            "share_of_step": float(level_ms.sum() / sum(serial_ms)),
            "serialised_step_ms": float(np.mean(serial_ms)),
            "bounds_kernel_avg_ms": float(bounds_ms.sum() / (args.steps * net.num_levels)),
        },
        "e2e": None if e2e_value is None else ({
            "value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "path": "gatspi_load_waveforms (each rank's windows from pinned host memory) + gatspi_simulate + "
                    "gatspi_toggle_stats_host + one int64 all-reduce of TC/T1 over the ranks"} if world > 1 else {
            "value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "path": "gatspi_load_testbench (whole-testbench waveforms from pinned host memory, cut into windows "
                    "on the GPU) + gatspi_simulate + gatspi_toggle_stats_host",
            "windowed_inputs": {"value": e2e_win[0], "h2d_bytes_per_step": int(e2e_win[1]),
                                "path": "gatspi_load_waveforms (host-cut windows) + simulate + toggle_stats_host"}}),
        "testbench_cut": cut,
        "gpu_launches": int(args.steps * launches_per_step),   # planning (non-empty levels), placement, simulation
        "clocks": clocks.summary(),
    }
    if world > 1:                      # the run's result: the statistics summed over the ranks
        tc_all, _ = shard.sum_stats(dist, tc, t1)
        line["events_all_ranks_per_step"] = int(tc_all.sum())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sim.close()
        line["cpu_baseline"] = cpu_baseline(net, stim, pulse_percent=args.pulse_percent)
    if rank == 0 and world == 1 and not args.no_e2e:
        line["sdf_translate"] = _sdf_translate(not args.no_cpu_baseline)
    if rank == 0:
        print(json.dumps(line))
    sim.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--pulse-percent", type=int, default=100,
                    help="PATHPULSEPERCENT of both inertial filters (100 = the page's setting, 0 = transport)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOAD_NAMES),
                    help="the workload timed (the 1M-gate configuration by default)")
    ap.add_argument("--pool-gb", type=float, default=0.0, help="waveform pool (0: sized for the workload)")
    ap.add_argument("--compact", action="store_true",
                    help="pack every level to its exact size after simulating it (GATSPI_FLAG_COMPACT)")
    ap.add_argument("--whole-windows", action="store_true",
                    help="never cut a window into time chunks (GATSPI_FLAG_WHOLE_WINDOWS; matters at 16 windows "
                         "or fewer)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--windows", type=int, default=0, help="profiling only: number of cycle windows")
    ap.add_argument("--cycles", type=int, default=0, help="profiling only: number of stimulus cycles")
    ap.add_argument("--gates", type=int, default=0, help="profiling only: number of gates of the netlist")
    ap.add_argument("--dump-levels", default="", metavar="PATH",
                    help="profiling only: write the run's per-level demand bytes to PATH (JSON)")
    ap.add_argument("--sweep", default="", metavar="ACTIVITY:WINDOWS",
                    help="one point of the activity x windows sweep on the same netlist instead of the default")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
