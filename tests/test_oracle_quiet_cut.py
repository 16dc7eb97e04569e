"""The quiet-time cut behind the time-chunk kernels, checked on the oracle (CPU).

Algorithm 1 of the GATSPI page simulates a (gate, window) from the window's start.
The kernels for few long windows also start a gate's simulation in the middle of a
window, at a quiet time T: no input pin of the gate has a transition in
[T - M1, T + M2), where M1 = the largest wire delay of its pins (rise or fall) + the
largest finite delay of its table and M2 = that wire delay + 1.  The claim is that,
at any PATHPULSEPERCENT, the gate's run from T on then depends only on every pin's
value at T (the first two tests take 100, the third 75, 50 and 0).  In the oracle's own terms: the window simulated as two windows, [0, T)
and [T, L), the second starting from the pins' values at T, gives exactly the
single window's output, with the same value at T, the same entries on either side
(shifted by T), the same toggle count and the same time at 1.

The cases are random single gates: 1 to 4 pins, random truth tables, conditional
delays (each column of the table drawn on its own), zero delays included, and input
waveforms with isolated edges and narrow pulses (some narrower than the wire delay,
so that the interconnect filter swallows them).  The cuts are the first and last
quiet time of every quiet stretch, the places where a wrong margin shows first, plus
random times inside the stretches.

The same search with a margin cut short must find a counterexample: M1 without the
gate delay (an output entry still pending at T), M1 without the wire delay (an
arrival still on its way at T), and M2 = 0 (a transition at T itself).  So the test
tells a sufficient rule from an insufficient one.  M2 = 1 turns out to be enough as
well: the pulse around T is already wider than any wire delay through M1, so the
wire delay in the kernels' M2 only makes a few quiet times unusable.
"""
import numpy as np

import synth
from helpers import EOW, INF, changes, single_gate, value_at

LENGTH = 700          # window length of the single-window run


def _random_gate(rng):
    """A one-gate netlist with n pins, its wire delays and its gate delay table."""
    n = int(rng.integers(1, 5))
    while True:
        tt = synth.cells.random_truth_table(n, rng)
        if 0 < int(tt.sum()) < tt.size:            # not a constant: the output moves
            break
    gmax = int(rng.choice([0, 3, 12, 40]))
    D = rng.integers(0 if gmax < 3 else 1, gmax + 1, size=(4 * n, 1 << (n - 1))).astype(np.int64)
    D[~synth.possible_rows(tt, n), :] = INF        # arcs the truth table cannot take
    wmax = int(rng.choice([0, 2, 9, 25]))
    rise = rng.integers(0, wmax + 1, size=n)
    fall = rng.integers(0, wmax + 1, size=n)
    net = single_gate(tt, n, D.astype(np.int32), wire_rise=rise, wire_fall=fall)
    return net, n, D, rise, fall


def _random_edges(rng):
    """Strictly increasing transition times in [1, LENGTH): isolated edges and pulses."""
    t = set()
    for _ in range(int(rng.integers(0, 12))):
        t.add(int(rng.integers(1, LENGTH)))
    for _ in range(int(rng.integers(0, 8))):     # pulses of width 1 .. 30
        a = int(rng.integers(1, LENGTH - 31))
        t.update((a, a + int(rng.integers(1, 31))))
    return sorted(t)


def _wave(init, edges):
    return ([-1, 0] if init else [0]) + list(edges) + [EOW]


def _quiet_times(edges_all, m1, m2, rng):
    """First and last quiet time of every quiet stretch, and a random one inside it:
    T in [m1 + 1, LENGTH) with no transition in [T - m1, T + m2)."""
    s = np.asarray(sorted(edges_all), np.int64)
    T = np.arange(m1 + 1, LENGTH, dtype=np.int64)
    inside = np.searchsorted(s, T + m2, side="left") - np.searchsorted(s, T - m1, side="left")
    quiet = T[inside == 0]
    if quiet.size == 0:
        return []
    brk = np.flatnonzero(np.diff(quiet) > 1)
    first = np.concatenate(([quiet[0]], quiet[brk + 1]))
    last = np.concatenate((quiet[brk], [quiet[-1]]))
    mid = [int(rng.integers(a, b + 1)) for a, b in zip(first, last)]
    return sorted(set(first.tolist()) | set(last.tolist()) | set(mid))


def _split_matches(oracle_lib, net, inits, edges, whole, T, pulse_percent=100):
    """Whether the window simulated as [0, T) and [T, LENGTH) equals the whole run."""
    waves = []
    for v0, e in zip(inits, edges):
        before = [t for t in e if t < T]
        after = [t - T for t in e if t > T]
        v_T = (v0 + sum(1 for t in e if t <= T)) % 2
        waves.append([_wave(v0, before), _wave(v_T, after)])
    two = oracle_lib.simulate(net, synth.from_waveforms(waves, [T, LENGTH - T]), pulse_percent=pulse_percent)
    out = whole.gate_wave(0, 0)
    a, b = two.gate_wave(0, 0), two.gate_wave(0, 1)
    return (value_at(a, 0) == value_at(out, 0) and value_at(b, 0) == value_at(out, T)
            and changes(a) + [t + T for t in changes(b)] == changes(out)
            and int(two.tc[0]) == int(whole.tc[0]) and int(two.t1[0]) == int(whole.t1[0]))


def test_quiet_cut_equals_whole_window(oracle_lib):
    """Cuts by the kernels' rule (and with M2 = 1) never change a gate's output; each
    shortened margin does."""
    rng = np.random.default_rng(2024)
    checked = 0
    wrong = {"rule": 0, "M1 without the gate delay": 0, "M1 without the wire delay": 0, "M2 = 0": 0}
    for case in range(600):
        net, n, D, rise, fall = _random_gate(rng)
        inits = [int(rng.integers(0, 2)) for _ in range(n)]
        edges = [_random_edges(rng) for _ in range(n)]
        whole = oracle_lib.simulate(net, synth.from_waveforms([[_wave(v, e)] for v, e in zip(inits, edges)],
                                                               LENGTH))
        wd = int(max(rise.max(), fall.max()))
        finite = D[D != INF]
        dg = int(finite.max()) if finite.size else 0
        rules = {"rule": (wd + dg, wd + 1), "M2 = 1": (wd + dg, 1), "M1 without the gate delay": (wd, wd + 1),
                 "M1 without the wire delay": (dg, wd + 1), "M2 = 0": (wd + dg, 0)}
        all_edges = [t for e in edges for t in e]
        for name, (m1, m2) in rules.items():
            for T in _quiet_times(all_edges, m1, m2, rng):
                ok = _split_matches(oracle_lib, net, inits, edges, whole, T)
                if name in ("rule", "M2 = 1"):
                    assert ok, (name, case, T, inits, edges)
                    checked += name == "rule"
                elif not ok:
                    wrong[name] += 1
    assert checked > 3000, checked
    for name in ("M1 without the gate delay", "M1 without the wire delay", "M2 = 0"):
        assert wrong[name] > 0, (name, wrong)


def _split_many_matches(oracle_lib, net, inits, edges, whole, cuts):
    """Whether the window simulated as len(cuts) + 1 windows, split at every cut (each
    part starting from the pins' values at its cut), equals the whole run."""
    bounds = [0] + list(cuts) + [LENGTH]
    waves = []
    for v0, e in zip(inits, edges):
        parts = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            v_a = (v0 + sum(1 for t in e if t <= a)) % 2 if a else v0
            parts.append(_wave(v_a, [t - a for t in e if a < t < b]))
        waves.append(parts)
    many = oracle_lib.simulate(net, synth.from_waveforms(waves, np.diff(bounds)))
    out = whole.gate_wave(0, 0)
    joined = []
    for k, a in enumerate(bounds[:-1]):
        part = many.gate_wave(0, k)
        if value_at(part, 0) != value_at(out, a):
            return False
        joined += [t + a for t in changes(part)]
    return (joined == changes(out) and int(many.tc[0]) == int(whole.tc[0])
            and int(many.t1[0]) == int(whole.t1[0]))


def test_many_quiet_cuts_equal_whole_window(oracle_lib):
    """A window cut at up to 31 quiet times at once, the way 32 lanes cut it: lane k
    takes the first quiet time at or after k * L / 32 that lies before the next
    lane's start, and a lane that finds none leaves its stretch to the lane before."""
    rng = np.random.default_rng(77)
    windows = 0
    cuts_total = 0
    for case in range(300):
        net, n, D, rise, fall = _random_gate(rng)
        inits = [int(rng.integers(0, 2)) for _ in range(n)]
        edges = [_random_edges(rng) for _ in range(n)]
        whole = oracle_lib.simulate(net, synth.from_waveforms([[_wave(v, e)] for v, e in zip(inits, edges)],
                                                               LENGTH))
        wd = int(max(rise.max(), fall.max()))
        finite = D[D != INF]
        dg = int(finite.max()) if finite.size else 0
        m1, m2 = wd + dg, wd + 1
        s = np.asarray(sorted(t for e in edges for t in e), np.int64)
        cuts = []
        for k in range(1, 32):
            lo, hi = k * LENGTH // 32, (k + 1) * LENGTH // 32
            for T in range(max(lo, m1 + 1), hi):
                if np.searchsorted(s, T + m2, side="left") == np.searchsorted(s, T - m1, side="left"):
                    cuts.append(T)
                    break
        assert _split_many_matches(oracle_lib, net, inits, edges, whole, cuts), (case, cuts)
        windows += 1
        cuts_total += len(cuts)
    assert cuts_total > 20 * windows, (cuts_total, windows)


def test_quiet_cut_holds_below_pulse_percent_100(oracle_lib):
    """The same cut rule at PATHPULSEPERCENT 75, 50 and 0 (transport): the split window
    still equals the whole run.  A pulse around T is wider than any reject limit, and an
    event after T makes an entry at least M2 + 1 + its delay after the last entry before
    T, more than that delay's reject limit, so no entry before T is ever cancelled."""
    for q in (75, 50, 0):
        rng = np.random.default_rng(500 + q)
        checked = 0
        for case in range(150):
            net, n, D, rise, fall = _random_gate(rng)
            inits = [int(rng.integers(0, 2)) for _ in range(n)]
            edges = [_random_edges(rng) for _ in range(n)]
            stim = synth.from_waveforms([[_wave(v, e)] for v, e in zip(inits, edges)], LENGTH)
            whole = oracle_lib.simulate(net, stim, pulse_percent=q)
            wd = int(max(rise.max(), fall.max()))
            finite = D[D != INF]
            dg = int(finite.max()) if finite.size else 0
            for T in _quiet_times([t for e in edges for t in e], wd + dg, wd + 1, rng):
                assert _split_matches(oracle_lib, net, inits, edges, whole, T, pulse_percent=q), (q, case, T)
                checked += 1
        assert checked > 1000, (q, checked)
