"""Synthetic SDF text for a synthetic netlist.

Input generation only: the text describes the delays the generator drew (the
per-instance conditional delay tables and the interconnect delays), written as SDF
3.0 statements, so that an SDF-to-table translator can be fed and checked.  It
evaluates nothing.

Names: inputs are ports ``pi<k>``; gate g is instance ``g<g>`` of its cell type; a
cell's input pins are those of the library (``I0 .. I<n-1>`` for random cells) and
its output is ``Y``.

Statements (the GATSPI page, Fig. 4, shows the kind: an unconditional IOPATH per
pin edge plus COND IOPATHs for the columns that differ):
* per gate pin and input edge: an IOPATH whose (rise) (fall) values are the most
  frequent values of the two rows over the columns, then one COND IOPATH per
  column whose pair differs; a row that is INF everywhere is written ``()``; when
  both input edges carry identical rows and the text style allows it, a single
  IOPATH without an edge covers both;
* per fanin edge: an INTERCONNECT from the driver to the pin with (rise) (fall).
Values are written in the file's TIMESCALE (decimals when it is coarser than the
netlist's unit), single or as ``min:typ:max`` triples (typ the value), chosen per
gate from the seed;
conditions mix the spellings ``A==1'b1``, ``A===1'b0``, ``A``, ``!A``, ``~A`` and the
operators ``&&`` and ``&``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .cells import _CELL_FUNCS
from .netlist import INF

_FS = {"s": 10**15, "ms": 10**12, "us": 10**9, "ns": 10**6, "ps": 10**3, "fs": 1}


@dataclass
class SdfText:
    text: str
    instance_names: list     # [G]
    input_names: list        # [P]
    pin_names: list          # per type: tuple of input pin names
    out_pin: str
    unit_fs: int             # the netlist's time unit in femtoseconds


def cell_pins(type_name: str, n: int) -> tuple:
    if type_name in _CELL_FUNCS:
        return _CELL_FUNCS[type_name][0]
    return tuple("I%d" % i for i in range(n))


def _num(v: int, scale: int) -> str:
    """v netlist units written in file units (scale netlist units per file unit)."""
    if scale == 1:
        return "%d" % v
    whole, frac = divmod(v, scale)
    return "%d.%0*d" % (whole, len(str(scale)) - 1, frac)


def _fmt(v: int, style: int, rng, scale: int) -> str:
    """One delay value: ``()`` for no arc, else a single value or a min:typ:max triple."""
    if v == INF:
        return "()"
    if style == 1:
        lo = max(0, v - int(rng.integers(0, 3)))
        return "(%s:%s:%s)" % (_num(lo, scale), _num(v, scale), _num(v + int(rng.integers(0, 3)), scale))
    return "(%s)" % _num(v, scale)


def _cond(names, bits, rng) -> str:
    terms = []
    for name, b in zip(names, bits):
        k = int(rng.integers(0, 4))
        if k == 0:
            terms.append("%s==1'b%d" % (name, b))
        elif k == 1:
            terms.append("%s===1'b%d" % (name, b))
        elif k == 2:
            terms.append(name if b else "!%s" % name)
        else:
            terms.append("(%s == 1'b%d)" % (name, b) if b else "~%s" % name)
    op = (" && ", "&&", " & ")[int(rng.integers(0, 3))]
    return op.join(terms)


def write_sdf(net, seed: int = 0, design: str = "top", file_unit: str = "1ps", unit_fs: int = 1000) -> SdfText:
    """SDF text of ``net``'s delays.  The netlist's integer delays are in units of
    ``unit_fs`` femtoseconds; ``file_unit`` is the file's TIMESCALE (a coarser unit
    makes the decimal style appear)."""
    rng = np.random.default_rng(seed)
    num = int("".join(c for c in file_unit if c.isdigit()) or "1")
    file_fs = num * _FS[file_unit.lstrip("0123456789").strip()]
    if file_fs % unit_fs or file_fs < unit_fs or len(str(file_fs // unit_fs).rstrip("0")) != 1:
        raise ValueError("the file unit must be a power-of-ten multiple of the netlist unit")
    scale = file_fs // unit_fs
    P, G = net.num_inputs, net.num_gates
    inst = ["g%d" % g for g in range(G)]
    inputs = ["pi%d" % p for p in range(P)]
    pins = [cell_pins(net.type_names[t], int(net.type_num_pins[t])) for t in range(len(net.type_names))]
    out = ['(DELAYFILE', ' (SDFVERSION "3.0")', ' (DESIGN "%s")' % design, ' (TIMESCALE %s)' % file_unit]

    def value(v, style):
        return _fmt(int(v), style, rng, scale)

    # interconnects, in the top cell
    wires = []
    fo = net.fanin_off
    for g in range(G):
        pn = pins[int(net.gate_type[g])]
        for i in range(int(fo[g + 1] - fo[g])):
            e = int(fo[g] + i)
            s = int(net.fanin_net[e])
            src = inputs[s] if s < P else "%s/Y" % inst[s - P]
            style = int(rng.integers(0, 2))
            wires.append('   (INTERCONNECT %s %s/%s %s %s)' % (src, inst[g], pn[i],
                                                             value(net.wire_rise[e], style),
                                                             value(net.wire_fall[e], style)))
    out.append(' (CELL (CELLTYPE "%s") (INSTANCE)' % design)
    out.append('  (DELAY (ABSOLUTE')
    out += wires
    out.append('  )))')

    for g in range(G):
        t = int(net.gate_type[g])
        n = int(net.type_num_pins[t])
        cols = 1 << (n - 1)
        D = np.asarray(net.dly_data[net.gate_dly_off[g]:net.gate_dly_off[g] + 4 * n * cols]).reshape(4 * n, cols)
        style = int(rng.integers(0, 2))
        out.append(' (CELL (CELLTYPE "%s") (INSTANCE %s)' % (net.type_names[t], inst[g]))
        out.append('  (DELAY (ABSOLUTE')
        for i in range(n):
            others = [pins[t][j] for j in range(n) if j != i]
            rows = {e_in: (D[4 * i + 2 * e_in + 0], D[4 * i + 2 * e_in + 1]) for e_in in (0, 1)}
            both = (np.array_equal(rows[0][0], rows[1][0]) and np.array_equal(rows[0][1], rows[1][1])
                    and rng.random() < 0.5)
            for e_in in ((None,) if both else (0, 1)):
                rr, rf = rows[0 if e_in is None else e_in]
                port = pins[t][i] if e_in is None else "(%s %s)" % ("posedge" if e_in == 0 else "negedge", pins[t][i])
                vals, counts = np.unique(np.stack([rr, rf], 1), axis=0, return_counts=True)
                mr, mf = (int(x) for x in vals[np.argmax(counts)])
                out.append('   (IOPATH %s Y %s %s)' % (port, value(mr, style), value(mf, style)))
                for c in range(cols):
                    if int(rr[c]) == mr and int(rf[c]) == mf:
                        continue
                    bits = [(c >> (n - 2 - k)) & 1 for k in range(n - 1)]
                    out.append('   (COND %s (IOPATH %s Y %s %s))' % (_cond(others, bits, rng), port,
                                                                     value(rr[c], style), value(rf[c], style)))
        out.append('  )))')
    out.append(')')
    return SdfText(text="\n".join(out) + "\n", instance_names=inst, input_names=inputs, pin_names=pins,
                   out_pin="Y", unit_fs=unit_fs)
