"""Pins of the oracle's SDF-to-delay-table translation (GATSPI page, Section 3, Fig. 4).

* Fig. 4's AOI21 statements give the printed B -> Y rows, the COND landing in the
  column of its condition (tests/golden/fig4_lookup.json);
* the synthetic SDF writer renders the generator's own delay tables and wire delays
  as text in several time scales and spellings: translating it back gives them
  exactly;
* hand-worked statements for every rule: edges, one value for both output edges,
  empty values, min:typ:max, COND over the unconditional whatever the order, the last
  COND where several hold, conversion and rounding, the default TIMESCALE,
  INTERCONNECT, errors.
"""
import json
import os

import numpy as np
import pytest

import synth
from helpers import INF

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _design(cells):
    """cells: list of (instance, type name, pin names); one gate each, tables packed."""
    type_names, type_pins, gate_type, inst, dly_off = [], [], [], [], []
    off = 0
    fanin = [0]
    for name, tname, pins in cells:
        if tname not in type_names:
            type_names.append(tname)
            type_pins.append(tuple(pins))
        gate_type.append(type_names.index(tname))
        inst.append(name)
        dly_off.append(off)
        n = len(pins)
        off += 4 * n * (1 << (n - 1))
        fanin.append(fanin[-1] + n)
    return dict(type_names=type_names, type_pins=type_pins, gate_type=np.array(gate_type),
                instance_names=inst, fanin_off=np.array(fanin), gate_dly_off=np.array(dly_off), dly_len=off)


def translate(sdf_mod, text, cells, unit_fs=1000):
    d = _design(cells)
    return sdf_mod.annotate(text, d["type_names"], d["type_pins"], d["gate_type"], d["instance_names"], d["fanin_off"],
                            d["gate_dly_off"], d["dly_len"], unit_fs)


def table(dly, n, first=0):
    cols = 1 << (n - 1)
    return dly[first:first + 4 * n * cols].reshape(4 * n, cols).tolist()


def _wrap(body, timescale="(TIMESCALE 1ps)"):
    return '(DELAYFILE (SDFVERSION "3.0") %s %s)' % (timescale, body)


AOI21 = ("A1", "A2", "B")


def fig4_text():
    fx = json.load(open(os.path.join(GOLDEN, "fig4_lookup.json")))["aoi21_B_to_Y"]
    stmts = []
    for key, rf in fx["sdf"].items():
        v = lambda x: "()" if x is None else "(%d)" % x            # noqa: E731
        path = key.split("IOPATH ")[1].rsplit(" Y", 1)[0]
        s = "(IOPATH %s Y %s %s)" % (path, v(rf["rise"]), v(rf["fall"]))
        if key.startswith("COND"):
            cond = key[len("COND "):key.index(" IOPATH")]
            s = "(COND %s %s)" % (cond, s)
        stmts.append(s)
    return fx, _wrap('(CELL (CELLTYPE "AOI21") (INSTANCE u1) (DELAY (ABSOLUTE %s)))' % " ".join(stmts))


def test_fig4_aoi21(oracle_sdf):
    fx, text = fig4_text()
    dly, _, _ = translate(oracle_sdf, text, [("u1", "AOI21", AOI21)])
    D = table(dly, 3)
    B = 2
    rows = fx["rows_printed"]
    assert D[4 * B + 2 * 1 + 0] == rows["B fall -> Y rise"]        # e_in FALL, e_out RISE
    assert D[4 * B + 2 * 0 + 1] == rows["B rise -> Y fall"]        # e_in RISE, e_out FALL
    assert D[4 * B + 0] == [INF] * 4 and D[4 * B + 3] == [INF] * 4
    assert rows["B fall -> Y rise"][fx["column_of_condition"]] == 7
    for r in range(8):                                             # A1, A2: no statements
        assert D[r] == [INF] * 4


@pytest.mark.parametrize("file_unit", ["1ps", "1ns", "10ps", "100ps"])
def test_round_trip_tiny(oracle_sdf, file_unit):
    net, _ = synth.make("tiny")
    s = synth.write_sdf(net, seed=len(file_unit), file_unit=file_unit)
    dly, wr, wf = oracle_sdf.annotate(s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names,
                                      net.fanin_off, net.gate_dly_off, net.dly_data.size, 1000)
    assert np.array_equal(dly, net.dly_data)
    assert np.array_equal(wr, net.wire_rise) and np.array_equal(wf, net.wire_fall)


@pytest.mark.parametrize("seed", range(4))
def test_round_trip_conditional_cells(oracle_sdf, seed):
    net = synth.generate_netlist(synth.NetlistSpec(
        num_gates=600, num_inputs=20, num_levels=5, seed=seed, cell_mix=(synth.CELL_MIX, ("random", 3))[seed % 2],
        cond_cells=("AOI21", "MUX2", "OAI22", "NAND4"), cond_fraction=0.6, delay_mode=("arc", "pin_out")[seed // 2]))
    s = synth.write_sdf(net, seed=seed, file_unit=("1ns", "1ps")[seed % 2])
    dly, wr, wf = oracle_sdf.annotate(s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names,
                                      net.fanin_off, net.gate_dly_off, net.dly_data.size, 1000)
    assert np.array_equal(dly, net.dly_data)
    assert np.array_equal(wr, net.wire_rise) and np.array_equal(wf, net.wire_fall)


# ---- hand-worked statements (shared with the library's translator tests) ----------

NAND2 = [("u", "NAND2", ("A", "B"))]


def _cell(body, tname="NAND2", inst="u"):
    return '(CELL (CELLTYPE "%s") (INSTANCE %s) (DELAY (ABSOLUTE %s)))' % (tname, inst, body)


# (text, cells, expected table of gate 0 as rows, or None) -- columns: the other pin
HAND = {
    # posedge sets e_in = RISE rows, negedge e_in = FALL, r = output rise, f = output fall
    "edges": (_wrap(_cell("(IOPATH (posedge A) Y (3) (4)) (IOPATH (negedge A) Y (5) (6))")), NAND2,
              [[3, 3], [4, 4], [5, 5], [6, 6]] + [[INF, INF]] * 4),
    # a bare pin sets both input edges; one value serves both output edges; () is no arc
    "bare pin, one value, empty": (_wrap(_cell("(IOPATH A Y (7)) (IOPATH B Y () (2))")), NAND2,
                                   [[7, 7]] * 4 + [[INF, INF], [2, 2], [INF, INF], [2, 2]]),
    # COND written before the unconditional statement still overrides it; columns are B's value
    "cond first": (_wrap(_cell("(COND B==1'b1 (IOPATH (posedge A) Y (9) (9))) (IOPATH (posedge A) Y (1) (2))")),
                   NAND2, [[1, 9], [2, 9]] + [[INF, INF]] * 6),
    # where two CONDs hold, the last one written wins
    "last cond": (_wrap(_cell("(IOPATH (negedge A) Y (1) (1)) (COND B (IOPATH (negedge A) Y (5) (5))) "
                              "(COND !B || B (IOPATH (negedge A) Y (6) ()))")), NAND2,
                  [[INF, INF]] * 2 + [[6, 6], [INF, INF]] + [[INF, INF]] * 4),
    # min:typ:max gives typ; a named condition
    "triple, named cond": (_wrap(_cell('(IOPATH (posedge B) Y (1:2:3) (4:5:6)) '
                                       '(COND "c0" ~A (IOPATH (posedge B) Y (7:8:9) (1:1:1)))')), NAND2,
                           [[INF, INF]] * 4 + [[8, 2], [1, 5]] + [[INF, INF]] * 2),
    # 1 ns file unit into 1 ps: 0.0125 -> 12.5 -> 13 (halves up), 0.0124 -> 12, 1.5e-2 -> 15
    "rounding": (_wrap(_cell("(IOPATH (posedge A) Y (0.0125) (0.0124)) (IOPATH (negedge A) Y (1.5e-2) (0))"),
                       "(TIMESCALE 1ns)"), NAND2, [[13, 13], [12, 12], [15, 15], [0, 0]] + [[INF, INF]] * 4),
    # no TIMESCALE: 1 ns
    "default timescale": ('(DELAYFILE %s)' % _cell("(IOPATH (posedge A) Y (2) (3))"), NAND2,
                          [[2000, 2000], [3000, 3000]] + [[INF, INF]] * 6),
    # a 3-pin condition over two other pins: columns (A1, A2), A1 most significant
    "two side pins": (_wrap(_cell("(IOPATH (posedge B) Y () (6)) (COND A1==1'b0 && A2===1'b1 (IOPATH (posedge B) Y "
                                  "() (5))) (COND (A1 & A2) | 0 (IOPATH (posedge B) Y () (4)))", "AOI21", "u")),
                      [("u", "AOI21", AOI21)],
                      [[INF] * 4] * 8 + [[INF] * 4, [6, 5, 6, 4], [INF] * 4, [INF] * 4]),
}

ERRORS = {
    "unknown instance": _wrap(_cell("(IOPATH A Y (1))", inst="nope")),
    "wrong celltype": _wrap(_cell("(IOPATH A Y (1))", tname="NOR2")),
    "condition on the switching pin": _wrap(_cell("(COND A (IOPATH (posedge A) Y (1)))")),
    "negative delay": _wrap(_cell("(IOPATH A Y (-1))")),
    "unbalanced": _wrap(_cell("(IOPATH A Y (1)")),
    "unknown pin": _wrap(_cell("(IOPATH C Y (1))")),
    "bad condition": _wrap(_cell("(COND B == (IOPATH (posedge A) Y (1)))")),
    "increment delays": _wrap('(CELL (CELLTYPE "NAND2") (INSTANCE u) (DELAY (INCREMENT (IOPATH A Y (1)))))'),
}


@pytest.mark.parametrize("name", sorted(HAND))
def test_hand_statements(oracle_sdf, name):
    text, cells, want = HAND[name]
    dly, _, _ = translate(oracle_sdf, text, cells)
    assert table(dly, len(cells[0][2])) == want


def test_interconnect(oracle_sdf):
    text = _wrap('(CELL (CELLTYPE "top") (INSTANCE) (DELAY (ABSOLUTE (INTERCONNECT pi0 u/B (3) (4)) '
                 '(INTERCONNECT x u/A (0:5:9)))))' + _cell("(IOPATH A Y (1))"))
    _, wr, wf = translate(oracle_sdf, text, NAND2)
    assert wr.tolist() == [5, 3] and wf.tolist() == [5, 4]


@pytest.mark.parametrize("name", sorted(ERRORS))
def test_errors(oracle_sdf, name):
    with pytest.raises(oracle_sdf.SdfError):
        translate(oracle_sdf, ERRORS[name], NAND2)


@pytest.fixture(scope="module")
def oracle_sdf():
    from oracle import sdf
    return sdf
