"""Pins of the CPU oracle to the worked examples the GATSPI page prints.

Fixtures in tests/golden/ hold the page's values with their citations:
* fig3_waveforms.json -- GATSPI page, Section 3, Fig. 3 (array format);
* fig4_lookup.json    -- GATSPI page, Section 3, Fig. 4 (truth table, SDF delay LUT).
The PATHPULSEPERCENT examples at the end are worked by hand from the rule the page
states (derivations beside them).
"""
import json
import os

import numpy as np
import pytest

import synth
from helpers import EOW, INF, changes, single_gate, uniform_delays, value_at

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _run(oracle_lib, net, waves, window_len):
    stim = synth.from_waveforms([[w] for w in waves], window_len)
    return oracle_lib.simulate(net, stim)


def test_fig3_format_through_buffer_and_inverter(oracle_lib):
    fx = _load("fig3_waveforms.json")
    for key in ("A", "B"):
        wave = fx[key]["printed"] + [fx["EOW"]]
        assert value_at(wave, 0) == fx[key]["initial_value"]
        for t, v in fx[key]["values_at"]:
            assert value_at(wave, t) == v
        # a zero-delay buffer reproduces the array; an inverter flips the head
        buf = single_gate(synth.truth_table("BUF"), 1, uniform_delays(1, 0, 0))
        r = _run(oracle_lib, buf, [wave], 200)
        assert r.gate_wave(0, 0).tolist() == wave
        inv = single_gate(synth.truth_table("INV"), 1, uniform_delays(1, 0, 0))
        r = _run(oracle_lib, inv, [wave], 200)
        out = r.gate_wave(0, 0).tolist()
        assert changes(out) == changes(wave)
        assert value_at(out, 0) == 1 - fx[key]["initial_value"]
        for t, v in fx[key]["values_at"]:
            assert value_at(out, t) == 1 - v


def test_fig3_time_at_one():
    """T1 of example A over [0, 200): value 1 on [0, 34) and [59, 123)."""
    import oracle
    fx = _load("fig3_waveforms.json")
    wave = fx["A"]["printed"] + [fx["EOW"]]
    buf = single_gate(synth.truth_table("BUF"), 1, uniform_delays(1, 0, 0))
    r = oracle.simulate(buf, synth.from_waveforms([[wave]], 200))
    assert int(r.t1[0]) == 34 + (123 - 59)
    assert int(r.t0[0]) == 200 - 98
    assert int(r.tc[0]) == 3


def test_fig4_nand2_index_and_value(oracle_lib):
    fx = _load("fig4_lookup.json")["nand2"]
    tt = np.array(fx["truth_table"], np.uint8)
    assert synth.truth_table("NAND2").tolist() == fx["truth_table"]
    ex = fx["example"]
    idx = ex["A"] * fx["pin_weights"]["A"] + ex["B"] * fx["pin_weights"]["B"]
    assert idx == ex["index"] and tt[idx] == ex["Y"]
    net = single_gate(tt, 2, uniform_delays(2, 3, 5, tt))
    assert net.pin_weight.tolist() == [fx["pin_weights"]["A"], fx["pin_weights"]["B"]]
    # A rises at 10, B at 20: the output (1 at start) falls when both are 1, 5 units later
    r = _run(oracle_lib, net, [[0, 10, EOW], [0, 20, EOW]], 100)
    assert r.gate_wave(0, 0).tolist() == [-1, 0, 25, EOW]


def _aoi21_table(fx):
    """AOI21 (A1, A2, B) delay table: B rows from the page, A1/A2 rows test-chosen."""
    tt = synth.truth_table("AOI21")
    n = 3
    D = np.full((4 * n, 4), 0, np.int64)
    for pin in (0, 1):                       # A1, A2: rise -> Y fall 30, fall -> Y rise 40
        for e_in in (0, 1):
            for e_out in (0, 1):
                D[4 * pin + 2 * e_in + e_out] = 30 if e_out == 1 else 40
    rows = fx["rows_printed"]
    D[4 * 2 + 2 * 1 + 0] = rows["B fall -> Y rise"]
    D[4 * 2 + 2 * 0 + 1] = rows["B rise -> Y fall"]
    ok = synth.possible_rows(tt, n)
    D[~ok] = INF
    # the page marks exactly the B rise->Y rise and B fall->Y fall rows impossible
    assert not ok[8] and ok[9] and ok[10] and not ok[11]
    return tt, D.astype(np.int32)


@pytest.mark.parametrize("a1,a2,expect", [
    (0, 1, [-1, 0, 105, 307]),   # COND A2==1 && A1==0 holds: column 1 -> 5 / 7
    (0, 0, [-1, 0, 106, 308]),   # plain IOPATH: 6 / 8
    (1, 0, [-1, 0, 106, 308]),
    (1, 1, [0]),                 # A1 & A2 hold Y at 0: B never changes it
])
def test_fig4_aoi21_conditional_delay(oracle_lib, a1, a2, expect):
    fx = _load("fig4_lookup.json")["aoi21_B_to_Y"]
    tt, D = _aoi21_table(fx)
    col = a1 * fx["side_pin_arc_weights"]["A1"] + a2 * fx["side_pin_arc_weights"]["A2"]
    assert (col == fx["column_of_condition"]) == (a1 == 0 and a2 == 1)
    net = single_gate(tt, 3, D, type_name="AOI21")
    static = lambda v: [-1, 0, EOW] if v else [0, EOW]  # noqa: E731
    r = _run(oracle_lib, net, [static(a1), static(a2), [0, 100, 300, EOW]], 1000)
    assert r.gate_wave(0, 0).tolist() == expect + [EOW]


def test_msi_takes_smallest_switching_arc(oracle_lib):
    """Both NAND2 inputs fall together: the output rises after the smaller arc delay
    (reading: IEEE 1364 shortest-path rule for simultaneous input changes)."""
    tt = synth.truth_table("NAND2")
    D = uniform_delays(2, 0, 0, tt).astype(np.int64)
    D[4 * 0 + 2 * 1 + 0] = 3     # A fall -> Y rise
    D[4 * 1 + 2 * 1 + 0] = 9     # B fall -> Y rise
    net = single_gate(tt, 2, D.astype(np.int32))
    r = _run(oracle_lib, net, [[-1, 0, 50, EOW], [-1, 0, 50, EOW]], 100)
    assert r.gate_wave(0, 0).tolist() == [0, 53, EOW]


def test_msi_skips_impossible_arc(oracle_lib):
    """f(A, B) = A: B has no arcs at all; A and B switching together uses A's arc."""
    tt = np.array([0, 0, 1, 1], np.uint8)
    D = uniform_delays(2, 7, 4, tt)
    assert (D[4:] == INF).all()
    net = single_gate(tt, 2, D)
    r = _run(oracle_lib, net, [[0, 50, 90, EOW], [-1, 0, 50, EOW]], 200)
    assert r.gate_wave(0, 0).tolist() == [0, 57, 94, EOW]


def test_missing_arc_is_an_error(oracle_lib):
    tt = np.array([0, 0, 1, 1], np.uint8)
    D = np.full((8, 2), INF, np.int32)
    net = single_gate(tt, 2, D)
    with pytest.raises(oracle_lib.OracleError) as e:
        _run(oracle_lib, net, [[0, 50, EOW], [0, EOW]], 100)
    assert e.value.code == 7


def test_malformed_input_is_an_error(oracle_lib):
    net = single_gate(synth.truth_table("BUF"), 1, uniform_delays(1, 1, 1))
    for bad in ([0, 5, 5, EOW], [0, 9, 3, EOW], [1, EOW], [0, 5], [-1, 3, EOW]):
        with pytest.raises(oracle_lib.OracleError) as e:
            _run(oracle_lib, net, [bad], 100)
        assert e.value.code == 4


# PATHPULSEPERCENT.  The GATSPI page (Section 3, the prose after Algorithm 1) fixes
# the pulse limit at 100 % of the delay and says other limits come from editing
# the gate filter's comparison.  Worked by hand from that rule, reading the limit as
# floor(delay * q / 100) in both the interconnect and the gate comparison:
#
# BUF, interconnect rise = fall = 4, gate delay 10 on both arcs; input pulses of
# widths 3, 7, 6, 14, 8, 12, 12 starting at 10.
#   q = 100: the interconnect drops [10, 13) (3 < 4); arrivals 24 30 44 52 64 76; the
#            gate (limit 10) cancels 34 at 30 (40 - 34 < 10) and 54 at 52, keeps 74, 86.
#   q = 50:  limits 2 and 5; every pulse reaches the pin: arrivals 14 17 24 30 44 52
#            64 76; 24 is cancelled at 17 (27 - 24 < 5); the rest stay.
#   q = 0:   nothing is filtered: every arrival + 10.
PULSE_WAVE = [0, 10, 13, 20, 26, 40, 48, 60, 72, EOW]
PULSE_EXPECT = {
    100: [0, 74, 86, EOW],
    50: [0, 34, 40, 54, 62, 74, 86, EOW],
    0: [0, 24, 27, 34, 40, 54, 62, 74, 86, EOW],
}

# BUF with a slow rise (10) and a fast fall (2), no interconnect delay; arrivals
# 5 7 20 21 22 31.  Each fall lands before the pending rise and cancels it, at any
# limit.  The last pair: the rise at 22 gives 32, the fall at 31 gives 33:
# 33 - 32 = 1 is below the q = 100 limit 2 (cancelled) but not below the q = 50
# limit 1 nor the q = 0 limit 0 (kept).
SKEW_WAVE = [0, 5, 7, 20, 21, 22, 31, EOW]
SKEW_EXPECT = {100: [0, EOW], 50: [0, 32, 33, EOW], 0: [0, 32, 33, EOW]}


@pytest.mark.parametrize("q", sorted(PULSE_EXPECT))
def test_pulse_percent_worked_example(oracle_lib, q):
    buf = single_gate(synth.truth_table("BUF"), 1, uniform_delays(1, 10, 10, synth.truth_table("BUF")),
                      wire_rise=[4], wire_fall=[4])
    r = oracle_lib.simulate(buf, synth.from_waveforms([[PULSE_WAVE]], 200), pulse_percent=q)
    assert r.gate_wave(0, 0).tolist() == PULSE_EXPECT[q]
    assert int(r.tc[0]) == len(PULSE_EXPECT[q]) - 2


@pytest.mark.parametrize("q", sorted(SKEW_EXPECT))
def test_pulse_percent_skewed_delays(oracle_lib, q):
    tt = synth.truth_table("BUF")
    buf = single_gate(tt, 1, uniform_delays(1, 10, 2, tt))
    r = oracle_lib.simulate(buf, synth.from_waveforms([[SKEW_WAVE]], 100), pulse_percent=q)
    assert r.gate_wave(0, 0).tolist() == SKEW_EXPECT[q]


def test_literal_single_pulse_test_study_variant(oracle_lib):
    """The interconnect pulse test read literally (one test per pin and event-loop
    iteration, the study variant) against the reading every other part takes (skip
    until the next pulse is wide enough).  A buffer (gate delay 1) behind a wire of
    delay 5; its input, at 0, toggles at 10, 12, 13, 15 and 100: two pulses of width 2
    back to back, then an edge, in a window of 200.
      reading taken: both pulses are skipped; 100 arrives at 105 and the output rises
        at 106: [0, 106, EOW], TC 1, T1 = 200 - 106 = 94;
      literal: the first iteration skips [10, 12) only and takes 13 (arriving at 18),
        so the output rises at 19; [15, 100) is wide, 15 arrives at 20 and the output
        falls at 21 (21 - 19 = 2 is not below the gate delay 1, so it is kept); 100
        gives 106: [0, 19, 21, 106, EOW], TC 3, T1 = 2 + 94 = 96."""
    buf = single_gate(np.array([0, 1], np.uint8), 1, uniform_delays(1, 1, 1), wire_rise=[5], wire_fall=[5])
    stim = synth.from_waveforms([[[0, 10, 12, 13, 15, 100, EOW]]], 200)
    taken = oracle_lib.simulate(buf, stim)
    literal = oracle_lib.simulate(buf, stim, literal_skip=True)
    assert taken.gate_wave(0, 0).tolist() == [0, 106, EOW]
    assert (int(taken.tc[0]), int(taken.t1[0])) == (1, 94)
    assert literal.gate_wave(0, 0).tolist() == [0, 19, 21, 106, EOW]
    assert (int(literal.tc[0]), int(literal.t1[0])) == (3, 96)
    # the switch is cleared after the call: the next run takes the reading again
    assert oracle_lib.simulate(buf, stim).gate_wave(0, 0).tolist() == [0, 106, EOW]
