"""Standard-cell library used by the synthetic netlists.

Each cell is a Boolean function of n ordered pins.  Its truth table is stored as a
1-D array of 2**n output bits, indexed by the sum of the weights of the pins at 1,
with the first pin carrying the largest weight 2**(n-1) (GATSPI page, Fig. 4: for
NAND2 the translator gives pin A the weight 2**1 and pin B the weight 2**0, and
Y = [1, 1, 1, 0]).

This module only describes the cells as data; it evaluates nothing at simulation
time.
"""
from __future__ import annotations

import itertools

import numpy as np

# name -> (pin names, Boolean function of the pin values in pin order)
_CELL_FUNCS = {
    "INV": (("A",), lambda a: 1 - a),
    "BUF": (("A",), lambda a: a),
    "NAND2": (("A", "B"), lambda a, b: 1 - (a & b)),
    "NOR2": (("A", "B"), lambda a, b: 1 - (a | b)),
    "XOR2": (("A", "B"), lambda a, b: a ^ b),
    "AOI21": (("A1", "A2", "B"), lambda a1, a2, b: 1 - ((a1 & a2) | b)),
    "OAI22": (("A1", "A2", "B1", "B2"), lambda a1, a2, b1, b2: 1 - ((a1 | a2) & (b1 | b2))),
    "MUX2": (("I0", "I1", "S"), lambda i0, i1, s: i1 if s else i0),
    "NAND4": (("A", "B", "C", "D"), lambda a, b, c, d: 1 - (a & b & c & d)),
}

# The nine-cell mix of the 50k / 1M / 5M-gate workloads, in a fixed order.
CELL_MIX = ("INV", "BUF", "NAND2", "NOR2", "XOR2", "AOI21", "OAI22", "MUX2", "NAND4")
# Cells of the scan-style run (2-input only).
SCAN_MIX = ("NAND2", "NOR2", "XOR2")


def pin_names(cell: str) -> tuple:
    return _CELL_FUNCS[cell][0]


def num_pins(cell: str) -> int:
    return len(_CELL_FUNCS[cell][0])


def truth_table(cell: str) -> np.ndarray:
    """2**n output bits; entry k holds f(v_0, ..., v_{n-1}) with k = sum v_i * 2**(n-1-i)."""
    names, fn = _CELL_FUNCS[cell]
    n = len(names)
    tt = np.zeros(1 << n, dtype=np.uint8)
    for vals in itertools.product((0, 1), repeat=n):
        k = 0
        for v in vals:
            k = (k << 1) | v
        tt[k] = fn(*vals)
    return tt


def random_truth_table(n: int, rng: np.random.Generator) -> np.ndarray:
    """A random n-input truth table (each of the 2**n rows an independent fair bit)."""
    return rng.integers(0, 2, size=1 << n, dtype=np.uint8)
