"""Seeded synthetic netlists and stimuli for the gate-level re-simulator.

Inputs only: nothing here simulates.  Both the CPU oracle and the CUDA path take
their inputs from these generators.
"""
from .cells import CELL_MIX, SCAN_MIX, truth_table  # noqa: F401
from .netlist import INF, Netlist, NetlistSpec, build_netlist, generate_netlist, possible_rows  # noqa: F401
from .stimulus import (EOW, Stimulus, StimulusSpec, Testbench, from_waveforms, generate_stimulus,  # noqa: F401
                       generate_testbench, select_windows)
from .workloads import SWEEP_ACTIVITY, SWEEP_WINDOWS, WORKLOADS, make, sweep, testbench  # noqa: F401
from .sdf import SdfText, write_sdf  # noqa: F401
