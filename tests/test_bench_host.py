"""bench.py's host arithmetic on the CPU: the algorithmic bytes of a run (the roofline's
numerator: each consumed waveform read once per run, each output written once, 8 bytes
of window index per consumed (net, window) and per (gate, window), 16 bytes per gate
and per fanin edge) and the per-level demand bytes, on a netlist small enough to count
by hand."""
import numpy as np

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
