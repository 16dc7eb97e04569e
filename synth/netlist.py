"""Seeded synthetic levelised netlists in the array form the simulator consumes.

Net numbering: primary / pseudo-primary inputs are nets 0 .. P-1, and gate g drives
net P + g.  Gates are numbered in logic-level order, so ``level_offsets`` delimits
each level's gate range and every fanin of a gate comes from a strictly lower
level (the PIs count as level -1).

Delay tables follow the GATSPI page, Fig. 4: per gate instance a 2-D array
D[4n][2**(n-1)] of int32.  The row is ``4*pin + 2*e_in + e_out`` with RISE = 0 and
FALL = 1 (the page's row order is scrambled in the extracted text; this order is
the reading used throughout).  The column is the sum of arc weights of the
non-switching pins at 1, the remaining pins taken in pin order with the first
carrying 2**(n-2) and the last 2**0 (the page's AOI21 example gives A1 = 2**1 and
A2 = 2**0 for the B -> Y arc).  Arcs that the cell's function can never exercise
(for example a rising input of a negative-unate pin raising the output) are set
to INF = INT32_MAX for the whole row, as Fig. 4 shows for AOI21 B -> Y.

Generation readings (stated here because the workload descriptions leave them
open):
* levels have equal width (the first ``G mod L`` levels take one extra gate);
* a gate's first pin draws from the previous level (the PIs for level 0) so that
  the level structure is realised; its other pins draw from all nets of earlier
  levels, PIs included;
* ``fanin="uniform"`` draws sources uniformly; ``fanin="geometric"`` gives every net
  a target fanout from Geometric(mean 2.5, support >= 1) and draws sources with
  probability proportional to that target (with replacement);
* gate delays are either drawn per (pin, output edge) (``delay_mode="pin_out"``,
  as in the tiny workload's "per-arc rise/fall delays") or per (pin, input edge,
  output edge) (``delay_mode="arc"``); conditional cells draw every column of a
  possible row separately, other cells repeat the row's value across columns;
* interconnect delays are drawn per fanin edge, rise and fall separately.

The generator builds inputs only; it evaluates no waveform.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import cells as _cells

INF = np.int32(2**31 - 1)
RISE, FALL = 0, 1


@dataclass
class NetlistSpec:
    num_gates: int
    num_inputs: int
    num_levels: int
    seed: int
    cell_mix: tuple = _cells.CELL_MIX       # or ("random", n) for random n-input truth tables
    fanin: str = "geometric"                # "uniform" | "geometric"
    fanout_mean: float = 2.5
    gate_delay: tuple = (5, 60)             # inclusive range
    delay_mode: str = "arc"                 # "arc" | "pin_out"
    wire_delay: tuple = (0, 3)              # inclusive range
    cond_cells: tuple = ("AOI21", "MUX2")   # cells whose instances all get conditional arcs
    cond_fraction: float = 0.0              # extra: this fraction of all multi-input instances


@dataclass
class Netlist:
    num_inputs: int
    num_gates: int
    num_levels: int
    level_offsets: np.ndarray   # int32 [L+1]
    type_names: list
    type_num_pins: np.ndarray   # int32 [T]
    type_tt_off: np.ndarray     # int32 [T]
    tt_data: np.ndarray         # uint8 [sum 2**n]
    gate_type: np.ndarray       # int32 [G]
    fanin_off: np.ndarray       # int32 [G+1]
    fanin_net: np.ndarray       # int32 [E]
    pin_weight: np.ndarray      # int32 [E]
    wire_rise: np.ndarray       # int32 [E]
    wire_fall: np.ndarray       # int32 [E]
    gate_dly_off: np.ndarray    # int64 [G]
    dly_data: np.ndarray        # int32 [...]
    stats: dict = field(default_factory=dict)

    @property
    def num_nets(self) -> int:
        return self.num_inputs + self.num_gates

    @property
    def num_edges(self) -> int:
        return int(self.fanin_off[-1])


def _possible_rows(tt: np.ndarray, n: int) -> np.ndarray:
    """bool[4n]: whether arc (pin i, e_in, e_out) can occur for this truth table."""
    ok = np.zeros(4 * n, dtype=bool)
    idx = np.arange(1 << n)
    for i in range(n):
        bit = 1 << (n - 1 - i)
        lo = idx[(idx & bit) == 0]          # rows with pin i at 0
        y0 = tt[lo]
        y1 = tt[lo | bit]
        for e_in in (RISE, FALL):
            before, after = (y0, y1) if e_in == RISE else (y1, y0)
            for e_out in (RISE, FALL):
                want = (0, 1) if e_out == RISE else (1, 0)
                ok[4 * i + 2 * e_in + e_out] = bool(np.any((before == want[0]) & (after == want[1])))
    return ok


def _level_sizes(num_gates: int, num_levels: int) -> np.ndarray:
    base, extra = divmod(num_gates, num_levels)
    sizes = np.full(num_levels, base, dtype=np.int64)
    sizes[:extra] += 1
    return sizes


def generate_netlist(spec: NetlistSpec) -> Netlist:
    rng = np.random.default_rng(spec.seed)
    G, P, L = spec.num_gates, spec.num_inputs, spec.num_levels
    if G < L:
        raise ValueError("need at least one gate per level")
    sizes = _level_sizes(G, L)
    level_offsets = np.zeros(L + 1, dtype=np.int64)
    level_offsets[1:] = np.cumsum(sizes)
    gate_level = np.repeat(np.arange(L), sizes)

    # ---- cell types -------------------------------------------------------
    if spec.cell_mix[0] == "random":
        n_rand = int(spec.cell_mix[1])
        tts = rng.integers(0, 2, size=(G, 1 << n_rand), dtype=np.uint8)
        keys = (tts.astype(np.int64) << np.arange(1 << n_rand)).sum(axis=1)
        uniq, gate_type = np.unique(keys, return_inverse=True)
        type_tts = [np.array([(int(k) >> b) & 1 for b in range(1 << n_rand)], dtype=np.uint8) for k in uniq]
        type_names = ["TT%d_%0*x" % (n_rand, (1 << n_rand) // 4 or 1, int(k)) for k in uniq]
        type_pins = [n_rand] * len(uniq)
    else:
        mix = tuple(spec.cell_mix)
        gate_type = rng.integers(0, len(mix), size=G)
        type_tts = [_cells.truth_table(c) for c in mix]
        type_names = list(mix)
        type_pins = [_cells.num_pins(c) for c in mix]
    gate_type = gate_type.astype(np.int32)
    T = len(type_names)
    type_num_pins = np.array(type_pins, dtype=np.int32)
    type_tt_off = np.zeros(T, dtype=np.int32)
    type_tt_off[1:] = np.cumsum([len(t) for t in type_tts])[:-1]
    tt_data = np.concatenate(type_tts).astype(np.uint8)

    # ---- fanin edges ------------------------------------------------------
    n_of_gate = type_num_pins[gate_type].astype(np.int64)
    fanin_off = np.zeros(G + 1, dtype=np.int64)
    fanin_off[1:] = np.cumsum(n_of_gate)
    E = int(fanin_off[-1])
    edge_gate = np.repeat(np.arange(G), n_of_gate)
    edge_pin = np.arange(E) - fanin_off[edge_gate]
    edge_level = gate_level[edge_gate]
    # net-id ranges: nets of level l are [P + level_offsets[l], P + level_offsets[l+1])
    net_start = np.concatenate(([0], P + level_offsets))     # start of "level" -1, 0, 1, ...
    first = edge_pin == 0
    lo = np.where(first, net_start[edge_level], 0)            # previous level, or all earlier nets
    hi = net_start[edge_level + 1]
    num_nets = P + G
    if spec.fanin == "uniform":
        fanin_net = lo + np.floor(rng.random(E) * (hi - lo)).astype(np.int64)
        fanin_net = np.minimum(fanin_net, hi - 1)
        target = None
    elif spec.fanin == "geometric":
        target = rng.geometric(1.0 / spec.fanout_mean, size=num_nets).astype(np.float64)
        cw = np.concatenate(([0.0], np.cumsum(target)))
        u = cw[lo] + rng.random(E) * (cw[hi] - cw[lo])
        fanin_net = np.searchsorted(cw, u, side="right") - 1
        fanin_net = np.clip(fanin_net, lo, hi - 1)
    else:
        raise ValueError(spec.fanin)
    fanin_net = fanin_net.astype(np.int32)
    pin_weight = (np.int64(1) << (n_of_gate[edge_gate] - 1 - edge_pin)).astype(np.int32)
    wlo, whi = spec.wire_delay
    wire_rise = rng.integers(wlo, whi + 1, size=E, dtype=np.int32)
    wire_fall = rng.integers(wlo, whi + 1, size=E, dtype=np.int32)

    # ---- per-instance delay tables -----------------------------------------
    rows_of_gate = 4 * n_of_gate
    cols_of_gate = np.int64(1) << (n_of_gate - 1)
    tbl = rows_of_gate * cols_of_gate
    gate_dly_off = np.zeros(G, dtype=np.int64)
    gate_dly_off[1:] = np.cumsum(tbl)[:-1]
    dly_data = np.empty(int(tbl.sum()), dtype=np.int32)
    dlo, dhi = spec.gate_delay
    multi = n_of_gate >= 2
    cond = np.zeros(G, dtype=bool)
    for t in range(T):
        if type_names[t] in spec.cond_cells:
            cond |= gate_type == t
    if spec.cond_fraction > 0:
        cond |= multi & (rng.random(G) < spec.cond_fraction)
    for t in range(T):
        gsel = np.nonzero(gate_type == t)[0]
        if gsel.size == 0:
            continue
        n = int(type_num_pins[t])
        R, C = 4 * n, 1 << (n - 1)
        c = gsel.size
        if spec.delay_mode == "pin_out":
            v = rng.integers(dlo, dhi + 1, size=(c, n, 2), dtype=np.int32)       # [gate, pin, e_out]
            r = np.arange(R)
            D = v[:, r // 4, r % 2][:, :, None].repeat(C, axis=2)
        elif spec.delay_mode == "arc":
            v = rng.integers(dlo, dhi + 1, size=(c, R, 1), dtype=np.int32)
            D = np.repeat(v, C, axis=2)
            csel = cond[gsel]
            if csel.any() and C > 1:
                D[csel] = rng.integers(dlo, dhi + 1, size=(int(csel.sum()), R, C), dtype=np.int32)
        else:
            raise ValueError(spec.delay_mode)
        ok = _possible_rows(type_tts[t], n)
        D[:, ~ok, :] = INF
        dst = gate_dly_off[gsel][:, None] + np.arange(R * C)[None, :]
        dly_data[dst.ravel()] = D.reshape(c, R * C).ravel()

    stats = {"edges": E, "cond_instances": int(cond.sum())}
    fo = np.bincount(fanin_net, minlength=num_nets)
    hist = np.bincount(np.minimum(fo, 20))
    stats["fanout_hist_0_to_20plus"] = hist.tolist()
    stats["fanout_mean_driven"] = float(fo[fo > 0].mean()) if (fo > 0).any() else 0.0
    stats["level_width"] = int(sizes.max())

    return Netlist(
        num_inputs=P, num_gates=G, num_levels=L,
        level_offsets=level_offsets.astype(np.int32),
        type_names=type_names, type_num_pins=type_num_pins, type_tt_off=type_tt_off,
        tt_data=tt_data, gate_type=gate_type,
        fanin_off=fanin_off.astype(np.int32), fanin_net=fanin_net, pin_weight=pin_weight,
        wire_rise=wire_rise, wire_fall=wire_fall,
        gate_dly_off=gate_dly_off, dly_data=dly_data, stats=stats,
    )


def build_netlist(num_inputs, level_gates, type_names, type_num_pins, type_tts,
                  gate_type, fanins, wire_rise, wire_fall, delay_tables) -> Netlist:
    """Assemble a small hand-written netlist (tests, worked examples).

    ``level_gates``: gates per level; ``fanins[g]``: list of source nets;
    ``delay_tables[g]``: array [4n][2**(n-1)].  Pin weights take the default
    first-pin-MSB convention.
    """
    G = len(gate_type)
    level_offsets = np.zeros(len(level_gates) + 1, dtype=np.int32)
    level_offsets[1:] = np.cumsum(level_gates)
    type_num_pins = np.asarray(type_num_pins, dtype=np.int32)
    type_tt_off = np.zeros(len(type_tts), dtype=np.int32)
    type_tt_off[1:] = np.cumsum([len(t) for t in type_tts])[:-1]
    fanin_off = np.zeros(G + 1, dtype=np.int32)
    fanin_off[1:] = np.cumsum([len(f) for f in fanins])
    n_of = [int(type_num_pins[t]) for t in gate_type]
    pin_weight = np.concatenate([[1 << (n - 1 - i) for i in range(n)] for n in n_of]).astype(np.int32)
    sizes = [np.asarray(d).size for d in delay_tables]
    gate_dly_off = np.zeros(G, dtype=np.int64)
    gate_dly_off[1:] = np.cumsum(sizes)[:-1]
    return Netlist(
        num_inputs=num_inputs, num_gates=G, num_levels=len(level_gates),
        level_offsets=level_offsets, type_names=list(type_names),
        type_num_pins=type_num_pins, type_tt_off=type_tt_off,
        tt_data=np.concatenate([np.asarray(t, dtype=np.uint8) for t in type_tts]),
        gate_type=np.asarray(gate_type, dtype=np.int32), fanin_off=fanin_off,
        fanin_net=np.concatenate([np.asarray(f, dtype=np.int32) for f in fanins]),
        pin_weight=pin_weight,
        wire_rise=np.asarray(wire_rise, dtype=np.int32).ravel(),
        wire_fall=np.asarray(wire_fall, dtype=np.int32).ravel(),
        gate_dly_off=gate_dly_off,
        dly_data=np.concatenate([np.asarray(d, dtype=np.int32).ravel() for d in delay_tables]),
    )


def possible_rows(tt, n) -> np.ndarray:
    """Public view of the impossible-arc mask used for INF rows (bool[4n])."""
    return _possible_rows(np.asarray(tt, dtype=np.uint8), int(n))
