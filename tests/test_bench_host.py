"""bench.py's host arithmetic on the CPU: the algorithmic bytes of a run (the roofline's
numerator: each consumed waveform read once per run, each output written once, 8 bytes
of window index per consumed (net, window) and per (gate, window), 16 bytes per gate
and per fanin edge) and the per-level demand bytes, on a netlist small enough to count
by hand."""
import json
import os

import numpy as np
import pytest

import bench
import synth
from helpers import uniform_delays


def _three_levels():
    """in0, in1 -> A = NAND2(in0, in1) (level 0) -> B = INV(A) (level 1) -> C = NAND2(A, B)
    (level 2): net A is consumed by two levels."""
    nand, inv = synth.truth_table("NAND2"), synth.truth_table("INV")
    return synth.build_netlist(num_inputs=2, level_gates=[1, 1, 1], type_names=["NAND2", "INV"],
                               type_num_pins=[2, 1], type_tts=[nand, inv], gate_type=[0, 1, 0],
                               fanins=[[0, 1], [2], [2, 3]], wire_rise=np.zeros(5), wire_fall=np.zeros(5),
                               delay_tables=[uniform_delays(2, 3, 4, nand), uniform_delays(1, 2, 2, inv),
                                             uniform_delays(2, 3, 4, nand)])


def test_algorithmic_bytes_by_hand():
    net = _three_levels()
    W = 2
    words = np.array([5, 7, 9, 4, 6])          # nets in0, in1, A, B, C over both windows
    total, parts = bench.algorithmic_bytes(net, words, W)
    # consumed nets: in0, in1 (by A), A (by B and C), B (by C) -- A once, not twice
    assert parts["read_waveforms"] == 4 * (5 + 7 + 9 + 4)
    assert parts["write_waveforms"] == 4 * (9 + 4 + 6)
    assert parts["window_index"] == 8 * W * (4 + 3)
    assert parts["descriptors"] == 16 * 3 + 16 * 5
    assert total == sum(parts.values()) == 100 + 76 + 112 + 128


def test_demand_bytes_by_hand():
    net = _three_levels()
    W = 2
    words = np.array([5, 7, 9, 4, 6])
    per_level = bench.demand_bytes(net, words, W)
    level0 = (4 * (5 + 7) + 8 * W * 2) + (4 * 9 + 8 * W) + (16 + 16 * 2)
    level1 = (4 * 9 + 8 * W) + (4 * 4 + 8 * W) + (16 + 16)
    level2 = (4 * (9 + 4) + 8 * W * 2) + (4 * 6 + 8 * W) + (16 + 16 * 2)   # A read again here
    assert per_level.tolist() == [level0, level1, level2]
    total, parts = bench.algorithmic_bytes(net, words, W)
    assert per_level.sum() > total     # demand counts A twice and every level's index again


def test_regime_picks_kernel_and_traffic_record(monkeypatch):
    """The roofline names the kernels that simulated the levels and scales its DRAM
    traffic from the ncu record of the same regime: windows ranked by bound (up to
    1024 windows), in window order (beyond), or cut into time chunks (no record);
    another PATHPULSEPERCENT or a record taken on other kernel code gives none."""
    import re
    with open(os.path.join(bench.ROOT, "gate_level_logic_gb300", "csrc", "gatspi_internal.cuh")) as f:
        lib_limit = int(re.search(r"kRankMaxWindows\s*=\s*(\d+)", f.read()).group(1))
    assert bench.RANKED_WINDOWS == lib_limit      # the same threshold as the library's planner
    assert bench.sim_regime(1, 1) == "ranked"
    assert bench.sim_regime(1, 256) == "ranked"
    assert bench.sim_regime(1, 1024) == "ranked"
    assert bench.sim_regime(1, 1025) == "window_order"
    assert bench.sim_regime(1, 4096) == "window_order"
    assert bench.sim_regime(32, 1) == "cut"
    assert bench.sim_regime(2, 16) == "cut"
    assert "level_chunk_kernel" in bench.SIM_REGIMES["cut"][0]
    ratios = {}
    for regime in ("ranked", "window_order"):
        traffic, ratio, name = bench._traffic(1e8, regime)
        with open(os.path.join(bench.ROOT, "profiles", name)) as f:
            rec = json.load(f)
        assert rec["kernel_sha"] == bench._kernel_hash()          # taken on the committed kernel code
        assert sum(x["dram_read"] + x["dram_write"] for x in rec["launches"]) == rec["dram_bytes"]
        assert sum(x["demand_bytes"] for x in rec["launches"]) == rec["demand_bytes"]
        assert ratio == pytest.approx(rec["dram_bytes"] / rec["demand_bytes"])
        assert traffic == pytest.approx(1e8 * ratio)
        ratios[regime] = ratio
    assert ratios["ranked"] != ratios["window_order"]
    assert bench._traffic(1e8, "cut") == (None, None, None)
    assert bench._traffic(1e8, "ranked", pulse_percent=60) == (None, None, None)
    monkeypatch.setattr(bench, "_kernel_hash", lambda: "0" * 16)
    assert bench._traffic(1e8, "window_order") == (None, None, None)
