"""Named synthetic workloads shaped like the GATSPI page's benchmarks (Table 2).

The page's own designs (NVDLA, industrial designs A-D, ICCAD2020 benchmarks) are not
available; these seeded stand-ins cover its ranges of size (1k - 2.3M gates),
activity (0.08 % - 120 %) and length (1.5k - 743k cycles).
"""
from __future__ import annotations

from .cells import CELL_MIX, SCAN_MIX
from .netlist import NetlistSpec, generate_netlist
from .stimulus import StimulusSpec, generate_stimulus, generate_testbench

# name -> (netlist spec kwargs, stimulus spec kwargs)
WORKLOADS = {
    # 200 random 2-input gates, 8 PIs, 4 levels; 100 cycles x period 100, p = 0.3; W = 1
    "tiny": (
        dict(num_gates=200, num_inputs=8, num_levels=4, seed=0, cell_mix=("random", 2),
             fanin="uniform", gate_delay=(1, 10), delay_mode="pin_out", wire_delay=(0, 3),
             cond_cells=()),
        dict(num_inputs=8, cycles=100, period=100, activity=0.3, windows=1, seed=0),
    ),
    # 50k gates, 20 levels, nine-cell mix; 256 PIs, 1000 cycles x 1000, 10 %; W = 16
    "50k": (
        dict(num_gates=50_000, num_inputs=256, num_levels=20, seed=1, cell_mix=CELL_MIX,
             fanin="geometric", gate_delay=(5, 60), delay_mode="arc", wire_delay=(0, 3),
             cond_cells=("AOI21", "MUX2")),
        dict(num_inputs=256, cycles=1000, period=1000, activity=0.10, windows=16, seed=1),
    ),
    # 1M gates, 40 levels; 4096 PIs, 10k cycles, 5 % with 10 % glitch pairs; W = 256
    "1M": (
        dict(num_gates=1_000_000, num_inputs=4096, num_levels=40, seed=2, cell_mix=CELL_MIX,
             fanin="geometric", gate_delay=(5, 60), delay_mode="arc", wire_delay=(0, 3),
             cond_cells=("AOI21", "MUX2")),
        dict(num_inputs=4096, cycles=10_000, period=1000, activity=0.05, windows=256, seed=2,
             glitch_frac=0.10, glitch_span=(1, 20)),
    ),
    # 5M gates, 60 levels, 30 % of multi-input cells conditional; 16k PIs, 2000 cycles, 20 %; W = 128
    "5M": (
        dict(num_gates=5_000_000, num_inputs=16_384, num_levels=60, seed=3, cell_mix=CELL_MIX,
             fanin="geometric", gate_delay=(5, 60), delay_mode="arc", wire_delay=(0, 3),
             cond_cells=(), cond_fraction=0.30),
        dict(num_inputs=16_384, cycles=2000, period=1000, activity=0.20, windows=128, seed=3),
    ),
    # scan-style run: 500k 2-input gates, 30 levels; 4096 PIs, 100k cycles at 2 %; W = 256
    "scan500k": (
        dict(num_gates=500_000, num_inputs=4096, num_levels=30, seed=4, cell_mix=SCAN_MIX,
             fanin="geometric", gate_delay=(5, 60), delay_mode="arc", wire_delay=(0, 3),
             cond_cells=()),
        dict(num_inputs=4096, cycles=100_000, period=1000, activity=0.02, windows=256, seed=4),
    ),
}

SWEEP_ACTIVITY = (0.01, 0.05, 0.20, 0.50)
SWEEP_WINDOWS = (1, 16, 256, 4096)


def make(name: str, **overrides):
    """(Netlist, Stimulus) of a named workload; ``overrides`` replace stimulus fields
    (e.g. ``activity``, ``windows``, ``cycles``) or, prefixed with ``net_``, netlist fields."""
    net_kw, stim_kw = (dict(d) for d in WORKLOADS[name])
    for k, v in overrides.items():
        if k.startswith("net_"):
            net_kw[k[4:]] = v
        else:
            stim_kw[k] = v
    net = generate_netlist(NetlistSpec(**net_kw))
    stim = generate_stimulus(StimulusSpec(**stim_kw))
    return net, stim


def testbench(name: str, **overrides):
    """The named workload's stimulus before the cut into windows (the same seeded edges
    as ``make``), for the testbench-restructuring path."""
    _, stim_kw = (dict(d) for d in WORKLOADS[name])
    stim_kw.update({k: v for k, v in overrides.items() if not k.startswith("net_")})
    return generate_testbench(StimulusSpec(**stim_kw))


def sweep(activity: float, windows: int):
    """One point of the 1M-gate sweep (seed 4 for the stimulus)."""
    return make("1M", activity=activity, windows=windows, seed=4, glitch_frac=0.0)
