"""Pins of the CPU oracle to closed forms, brute force and invariants.

* each library cell's lookup against its textbook Boolean function;
* the event-driven oracle against an independent unit-time-step simulator of
  inertial wire and gate elements, over many seeded tiny netlists;
* all-zero delays: every net equals the combinational function of the inputs;
* BUF / INV chains with equal rise and fall delay d: a delay line that drops every
  pulse shorter than d (inertial delay), or shorter than floor(d * q / 100) at
  PATHPULSEPERCENT q (q = 0: transport delay, nothing dropped);
* other PATHPULSEPERCENT values against the unit-step simulator, whose elements
  then hold queues of pending events;
* cycle windows: when every event settles inside its cycle, simulating W windows
  equals the single-window run cut at the window boundaries;
* format invariants of every output waveform and of the toggle statistics.
"""
import itertools

import numpy as np
import pytest

import synth
from helpers import EOW, changes, permute_pin_weights, single_gate, uniform_delays, value_at
from synth.netlist import NetlistSpec, generate_netlist
from synth.stimulus import StimulusSpec, generate_stimulus

CLOSED_FORM = {
    "INV": lambda a: 1 - a,
    "BUF": lambda a: a,
    "NAND2": lambda a, b: int(not (a and b)),
    "NOR2": lambda a, b: int(not (a or b)),
    "XOR2": lambda a, b: int(a != b),
    "AOI21": lambda a1, a2, b: int(not ((a1 and a2) or b)),
    "OAI22": lambda a1, a2, b1, b2: int(not ((a1 or a2) and (b1 or b2))),
    "MUX2": lambda i0, i1, s: i1 if s else i0,
    "NAND4": lambda a, b, c, d: int(not (a and b and c and d)),
}


def _vector_walk(n, seed):
    """Input vectors visiting every combination, in a shuffled order, plus a walk back."""
    rng = np.random.default_rng(seed)
    combos = list(itertools.product((0, 1), repeat=n))
    order = [combos[i] for i in rng.permutation(len(combos))]
    return order + order[::-1]


@pytest.mark.parametrize("cell", synth.CELL_MIX)
@pytest.mark.parametrize("delay", [0, 4])
def test_cell_matches_closed_form(oracle_lib, cell, delay):
    n = synth.cells.num_pins(cell)
    tt = synth.truth_table(cell)
    f = CLOSED_FORM[cell]
    net = single_gate(tt, n, uniform_delays(n, delay, delay, tt), type_name=cell)
    vecs = _vector_walk(n, seed=n)
    step = 10
    waves = []
    for i in range(n):
        w = [-1, 0] if vecs[0][i] else [0]
        for k in range(1, len(vecs)):
            if vecs[k][i] != vecs[k - 1][i]:
                w.append(k * step)
        waves.append(w + [EOW])
    stim = synth.from_waveforms([[w] for w in waves], step * (len(vecs) + 2))
    out = oracle_lib.simulate(net, stim).gate_wave(0, 0)
    for k, v in enumerate(vecs):
        assert value_at(out, k * step + delay) == f(*v), (cell, k, v)
    # no redundant entries: every change flips the closed-form value
    expect = [k * step + delay for k in range(1, len(vecs)) if f(*vecs[k]) != f(*vecs[k - 1])]
    assert changes(out) == expect


def _random_case(seed):
    rng = np.random.default_rng(10_000 + seed)
    mix = [("random", 2), ("random", 3), synth.CELL_MIX, ("random", 4), ("random", 1)][seed % 5]
    G = int(rng.integers(3, 80))
    L = min(int(rng.integers(1, 6)), G)
    wire = [(0, 3), (0, 1), (0, 0), (0, 6)][seed % 4]
    gate = [(0, 2), (1, 3), (1, 10), (5, 60), (0, 0)][seed % 5]
    if gate == (0, 0):
        wire = (0, 0)
    net = generate_netlist(NetlistSpec(
        num_gates=G, num_inputs=int(rng.integers(1, 8)), num_levels=L, seed=seed, cell_mix=mix,
        fanin=("uniform", "geometric")[seed % 2], gate_delay=gate, delay_mode=("arc", "pin_out")[seed % 2],
        wire_delay=wire, cond_cells=("AOI21", "MUX2"), cond_fraction=0.4))
    W = int(rng.integers(1, 4))
    stim = generate_stimulus(StimulusSpec(
        num_inputs=net.num_inputs, cycles=int(rng.integers(W, 25)), period=int(rng.integers(4, 40)),
        activity=float(rng.choice([0.1, 0.5, 0.9])), windows=W, seed=seed,
        glitch_frac=float(rng.choice([0.0, 0.4, 0.8])), glitch_span=(1, int(rng.integers(1, 8)))))
    return net, stim


@pytest.mark.parametrize("block", range(6))
def test_oracle_equals_bruteforce(oracle_lib, block):
    """300 seeded tiny netlists per block: waveforms, TC and T1 identical."""
    zero_width = 0
    for seed in range(block * 300, (block + 1) * 300):
        net, stim = _random_case(seed)
        r = oracle_lib.simulate(net, stim)
        b = oracle_lib.bruteforce(net, stim)
        assert np.array_equal(r.off, b.off), seed
        assert np.array_equal(r.pool, b.pool), seed
        assert np.array_equal(r.tc, b.tc), seed
        assert np.array_equal(r.t1, b.t1), seed
        body = r.pool[r.off[net.num_inputs * stim.num_windows]:]
        zero_width += int(np.sum((body[1:] == body[:-1]) & (body[1:] != EOW)))
    assert zero_width > 0     # the sample exercises equal-time edges on one pin


def test_tiny_workload_equals_bruteforce(oracle_lib):
    net, stim = synth.make("tiny")
    r = oracle_lib.simulate(net, stim)
    b = oracle_lib.bruteforce(net, stim)
    assert np.array_equal(r.pool, b.pool) and np.array_equal(r.tc, b.tc) and np.array_equal(r.t1, b.t1)


def _combinational(net, stim, t):
    """Value of every net at time t by plain level-order evaluation (window 0)."""
    P = net.num_inputs
    val = np.zeros(P + net.num_gates, np.int64)
    for s in range(P):
        val[s] = value_at(stim.window(s, 0), t)
    for g in range(net.num_gates):
        ty = net.gate_type[g]
        n = net.type_num_pins[ty]
        pins = net.fanin_net[net.fanin_off[g]:net.fanin_off[g] + n]
        k = int(sum(int(val[s]) * int(w) for s, w in zip(pins, net.pin_weight[net.fanin_off[g]:net.fanin_off[g] + n])))
        val[P + g] = net.tt_data[net.type_tt_off[ty] + k]
    return val


def test_zero_delay_equals_combinational(oracle_lib):
    net = generate_netlist(NetlistSpec(num_gates=300, num_inputs=12, num_levels=8, seed=7, cell_mix=synth.CELL_MIX,
                                       gate_delay=(0, 0), wire_delay=(0, 0), cond_cells=("AOI21", "MUX2")))
    stim = generate_stimulus(StimulusSpec(num_inputs=12, cycles=40, period=10, activity=0.4, windows=1, seed=7))
    r = oracle_lib.simulate(net, stim)
    times = sorted({int(x) for s in range(net.num_inputs) for x in changes(stim.window(s, 0))})
    prev = _combinational(net, stim, 0)
    expect = {g: [] for g in range(net.num_gates)}
    for t in times:
        cur = _combinational(net, stim, t)
        for g in np.nonzero(cur[net.num_inputs:] != prev[net.num_inputs:])[0]:
            expect[int(g)].append(t)
        prev = cur
    init = _combinational(net, stim, 0)
    for g in range(net.num_gates):
        out = r.gate_wave(g, 0)
        assert value_at(out, 0) == init[net.num_inputs + g]
        assert changes(out) == expect[g], g


def _inertial_closed_form(times, init, d, r=None):
    """Inertial delay d with pulse reject limit r (r = d unless given): an input change
    to v at t reaches the output at t + d when the input then holds v for at least r
    and v differs from the output."""
    r = d if r is None else r
    out, cur = [], init
    for k, t in enumerate(times):
        v = init ^ ((k + 1) & 1)
        nxt = times[k + 1] if k + 1 < len(times) else None
        if (nxt is None or nxt - t >= r) and v != cur:
            out.append(t + d)
            cur = v
    return out


@pytest.mark.parametrize("seed", range(8))
def test_buffer_inverter_chain_is_inertial_delay_line(oracle_lib, seed):
    rng = np.random.default_rng(seed)
    k = int(rng.integers(1, 7))
    d = int(rng.integers(1, 12))
    kinds = [("BUF", "INV")[int(b)] for b in rng.integers(0, 2, size=k)]
    types = ["BUF", "INV"]
    tts = [synth.truth_table(c) for c in types]
    net = synth.build_netlist(num_inputs=1, level_gates=[1] * k, type_names=types, type_num_pins=[1, 1],
                              type_tts=tts, gate_type=[types.index(c) for c in kinds],
                              fanins=[[g] for g in range(k)], wire_rise=np.zeros(k), wire_fall=np.zeros(k),
                              delay_tables=[uniform_delays(1, d, d, tts[types.index(c)]) for c in kinds])
    gaps = rng.integers(1, 3 * d + 1, size=60)
    times = np.cumsum(gaps).tolist()
    init = int(rng.integers(0, 2))
    wave = ([-1, 0] if init else [0]) + times + [EOW]
    r = oracle_lib.simulate(net, synth.from_waveforms([[wave]], times[-1] + 10 * k * d))
    stage1 = _inertial_closed_form(times, init, d)
    inv = 0
    for g in range(k):
        inv ^= kinds[g] == "INV"
        out = r.gate_wave(g, 0)
        assert changes(out) == [t + g * d for t in stage1]
        assert value_at(out, 0) == init ^ inv


@pytest.mark.parametrize("q", [100, 60, 25, 0])
@pytest.mark.parametrize("seed", range(6))
def test_chain_with_pulse_limit_is_filtered_delay_line(oracle_lib, q, seed):
    """PATHPULSEPERCENT q: every interconnect (rise = fall = dw) and every gate (delay d)
    of a BUF/INV chain is a delay line that drops the pulses narrower than its reject
    limit floor(delay * q / 100); q = 0 drops none (transport delay)."""
    rng = np.random.default_rng(500 + seed)
    k = int(rng.integers(1, 6))
    d = int(rng.integers(1, 14))
    dw = int(rng.integers(0, 7))
    kinds = [("BUF", "INV")[int(b)] for b in rng.integers(0, 2, size=k)]
    types = ["BUF", "INV"]
    tts = [synth.truth_table(c) for c in types]
    net = synth.build_netlist(num_inputs=1, level_gates=[1] * k, type_names=types, type_num_pins=[1, 1],
                              type_tts=tts, gate_type=[types.index(c) for c in kinds],
                              fanins=[[g] for g in range(k)], wire_rise=np.full(k, dw), wire_fall=np.full(k, dw),
                              delay_tables=[uniform_delays(1, d, d, tts[types.index(c)]) for c in kinds])
    times = np.cumsum(rng.integers(1, 2 * (d + dw) + 2, size=80)).tolist()
    wave = [0] + times + [EOW]
    r = oracle_lib.simulate(net, synth.from_waveforms([[wave]], times[-1] + 10 * k * (d + dw)), pulse_percent=q)
    cur = times
    for g in range(k):
        cur = _inertial_closed_form(cur, 0, dw, dw * q // 100)      # the gate's interconnect
        cur = _inertial_closed_form(cur, 0, d, d * q // 100)        # the gate
        assert changes(r.gate_wave(g, 0)) == cur, (q, seed, g)
    if q == 0:
        assert len(changes(r.gate_wave(k - 1, 0))) == len(times)


def _skew_free(net):
    """The same netlist with every interconnect's fall delay set to its rise delay."""
    net.wire_fall = net.wire_rise.copy()
    return net


@pytest.mark.parametrize("q", [0, 20, 50, 75, 99])
def test_oracle_equals_bruteforce_pulse_percent(oracle_lib, q):
    """Other PATHPULSEPERCENT values against the unit-step model with pending-event
    queues (interconnect rise = fall, so that no element's events fall due out of
    order); the sample must differ from the q = 100 result often."""
    differ = 0
    for seed in range(200):
        net, stim = _random_case(seed)
        net = _skew_free(net)
        r = oracle_lib.simulate(net, stim, pulse_percent=q)
        b = oracle_lib.bruteforce(net, stim, pulse_percent=q)
        assert np.array_equal(r.off, b.off), (q, seed)
        assert np.array_equal(r.pool, b.pool), (q, seed)
        assert np.array_equal(r.tc, b.tc) and np.array_equal(r.t1, b.t1), (q, seed)
        differ += not np.array_equal(r.pool, oracle_lib.simulate(net, stim).pool)
    assert differ >= 40


def test_oracle_equals_bruteforce_pulse_percent_skewed_wires(oracle_lib):
    """Interconnects with different rise and fall delays: every case the unit-step
    model can order (its events fall due in order) agrees with the oracle."""
    agree = 0
    for seed in range(300):
        net, stim = _random_case(seed)
        q = (0, 40, 80)[seed % 3]
        r = oracle_lib.simulate(net, stim, pulse_percent=q)
        try:
            b = oracle_lib.bruteforce(net, stim, pulse_percent=q)
        except oracle_lib.OracleError as e:
            assert "out of order" in str(e)
            continue
        assert np.array_equal(r.pool, b.pool) and np.array_equal(r.tc, b.tc) and np.array_equal(r.t1, b.t1), seed
        agree += 1
    assert agree >= 150


def test_pulse_percent_out_of_range_is_rejected(oracle_lib):
    net, stim = synth.make("tiny")
    for q in (-1, 101):
        with pytest.raises(oracle_lib.OracleError):
            oracle_lib.simulate(net, stim, pulse_percent=q)


def test_windows_equal_cut_single_run(oracle_lib):
    """Events settle within their cycle (offsets <= 100, longest path < 100, period 300):
    every window then starts from the previous window's settled state."""
    net = generate_netlist(NetlistSpec(num_gates=400, num_inputs=16, num_levels=6, seed=11,
                                       cell_mix=synth.CELL_MIX, gate_delay=(1, 10), wire_delay=(0, 3),
                                       cond_cells=("AOI21", "MUX2")))
    spec = dict(num_inputs=16, cycles=12, period=300, activity=0.5, seed=11, glitch_frac=0.3,
                glitch_span=(1, 8), max_offset=100)
    one = oracle_lib.simulate(net, generate_stimulus(StimulusSpec(windows=1, **spec)))
    for W in (2, 3, 4, 12):
        stim = generate_stimulus(StimulusSpec(windows=W, **spec))
        many = oracle_lib.simulate(net, stim)
        start = np.concatenate(([0], np.cumsum(stim.window_len)))
        for g in range(net.num_gates):
            full = one.gate_wave(g, 0)
            ch = np.array(changes(full), dtype=np.int64)
            for w in range(W):
                part = many.gate_wave(g, w)
                assert value_at(part, 0) == value_at(full, int(start[w])), (W, g, w)
                inside = ch[(ch >= start[w]) & (ch < start[w + 1])] - start[w]
                assert changes(part) == inside.tolist(), (W, g, w)
        assert np.array_equal(many.tc, one.tc)
        assert np.array_equal(many.t1, one.t1)


@pytest.mark.parametrize("name", ["tiny", "50k"])
def test_output_invariants(oracle_lib, name):
    net, stim = synth.make(name)
    r = oracle_lib.simulate(net, stim, threads=4)
    P, G, W = net.num_inputs, net.num_gates, stim.num_windows
    lens = np.diff(r.off)
    assert (lens >= 2).all() and r.off[0] == 0 and r.off[-1] == r.pool.size
    pool = r.pool.astype(np.int64)
    k = np.arange(P * W, (P + G) * W)                 # gate waveforms
    s, e = r.off[k], r.off[k + 1]
    assert (pool[e - 1] == EOW).all()
    head = np.where(pool[s] == -1, 2, 1)
    assert (pool[s + head - 1] == 0).all()
    # every entry after the first is larger than the one before (gate delays >= 1)
    owner = np.repeat(np.arange(k.size), e - s)
    pos = np.arange(int(s[0]), int(e[-1]))
    not_first = pos != s[owner]
    assert (pool[pos[not_first]] > pool[pos[not_first] - 1]).all()
    ntog = (e - s) - head - 1
    y_init, y_final = head - 1, (e - s - 2) % 2
    assert ((ntog % 2) == (y_init ^ y_final)).all()
    gate = (k - P * W) // W
    assert np.array_equal(np.bincount(gate, weights=ntog, minlength=G).astype(np.int64), r.tc)
    # time at 1 in [0, L): integrate every interval [entry, next entry) of value index % 2
    L = stim.window_len[(k - P * W) % W]
    last = pos == e[owner] - 1
    ent = pos[~last]
    o = owner[~last]
    lo = np.clip(pool[ent], 0, L[o])
    hi = np.clip(np.where(pos[~last] + 1 == e[o] - 1, L[o], pool[ent + 1]), 0, L[o])
    ones = np.where((ent - s[o]) % 2 == 1, hi - lo, 0)
    t1 = np.bincount(gate[o], weights=ones, minlength=G).astype(np.int64)
    assert np.array_equal(t1, r.t1)
    assert np.array_equal(r.t0 + r.t1, np.full(G, int(stim.window_len.sum())))


def test_threads_do_not_change_results(oracle_lib):
    net, stim = synth.make("50k")
    a = oracle_lib.simulate(net, stim, threads=1)
    b = oracle_lib.simulate(net, stim, threads=5)
    assert np.array_equal(a.off, b.off) and np.array_equal(a.pool, b.pool)
    assert np.array_equal(a.tc, b.tc) and np.array_equal(a.t1, b.t1)


def test_pin_weights_are_data(oracle_lib):
    """Permuting every gate's truth-table pin weights, with the table re-indexed to the
    same function, changes nothing (Fig. 4: weights come from the translator)."""
    net, stim = synth.make("tiny")
    perm = permute_pin_weights(net, seed=3)
    assert not np.array_equal(perm.pin_weight, net.pin_weight)
    a = oracle_lib.simulate(net, stim)
    b = oracle_lib.simulate(perm, stim)
    assert np.array_equal(a.pool, b.pool) and np.array_equal(a.tc, b.tc) and np.array_equal(a.t1, b.t1)


def _bound_slack(net, stim, r):
    """Per (gate, window): 3 + sum over pins of (source length - 2), minus the output's
    length (words, EOW included).  Each arrival step stores at most one entry, so a
    window's entries are at most its pins' transitions, at most (length - 2) each; the
    head takes one or two words and the EOW one."""
    P, G, W = net.num_inputs, net.num_gates, stim.num_windows
    lens = np.diff(r.off).reshape(P + G, W)
    pins = np.diff(net.fanin_off).astype(np.int64)
    gate_of_edge = np.repeat(np.arange(G), pins)
    src = lens[np.asarray(net.fanin_net, np.int64)] - 2                  # [E, W]
    per_gate = np.zeros((G, W), np.int64)
    np.add.at(per_gate, gate_of_edge, src)
    return 3 + per_gate - lens[P:]


def test_output_length_bound(oracle_lib):
    """Every output fits the bound its inputs' lengths give (the size of its slot before
    anything is simulated), and the bound is reached: a constant one word smaller
    would be exceeded, and one word larger would never be used."""
    cases = [_random_case(seed) for seed in range(600)] + [synth.make("tiny"), synth.make("50k")]
    tight = 0
    for net, stim in cases:
        slack = _bound_slack(net, stim, oracle_lib.simulate(net, stim, threads=4))
        assert slack.min() >= 0
        tight += int(np.sum(slack == 0))
    assert tight > 0
