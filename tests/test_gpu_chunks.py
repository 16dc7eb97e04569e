"""Windows cut into time chunks (16 windows or fewer, any PATHPULSEPERCENT): every
lane of a gate's warp simulates its window between two quiet times of the gate, and the
warp moves the chunks' entries together.  The waveforms, window offsets and TC/T0/T1
must equal the oracle's whole-window run bit for bit, whichever cuts are found, on the
corner cases the oracle was pinned on (zero delays, zero-width pulses, 1-4 pin random
cells, conditional arcs), on stretches too busy to hold a cut, on every launch path, with
packing, after a stalled scan, when a load switches a context between cut and whole
windows, and below PATHPULSEPERCENT 100."""
import os

import numpy as np
import pytest

import synth
from helpers import EOW, INF, single_gate
from test_gpu_parity import assert_same, pool_for, run_gpu

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def gpu():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    from gate_level_logic_gb300 import Simulator
    return Simulator


def flags():
    from gate_level_logic_gb300 import gatspi
    return gatspi.GATSPI_FLAG_CUT_WINDOWS, gatspi.GATSPI_FLAG_WHOLE_WINDOWS


def lanes(Simulator, net, stim, pool_words, fl):
    with Simulator(net, stim.window_len, pool_words=pool_words, flags=fl) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        return sim.lanes_per_window()


@pytest.mark.parametrize("W", [1, 2, 3, 5, 7, 8, 11, 16])
def test_cut_and_whole_windows_equal_the_oracle(gpu, oracle_lib, W):
    """Every window count that is cut (32 // W lanes per window, idle lanes when W does
    not divide 32), forced cut and forced whole, against the oracle."""
    cut, whole = flags()
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=3001, num_inputs=37, num_levels=9, seed=900 + W,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=37, cycles=2000, period=300, activity=0.3,
                                                      windows=W, seed=W, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    pw = pool_for(ref, net)
    assert lanes(gpu, net, stim, pw, cut) == 32 // W
    assert lanes(gpu, net, stim, pw, whole) == 1
    assert_same(run_gpu(gpu, net, stim, pw, flags=cut), ref, "cut W=%d" % W)
    assert_same(run_gpu(gpu, net, stim, pw, flags=whole), ref, "whole W=%d" % W)


def test_cut_windows_random_small_netlists(gpu, oracle_lib):
    """The 120 seeded corner-heavy cases (zero wire and gate delays, so margins of 0 and
    1; zero-width pulses; equal timestamps on one pin; conditional arcs; 1 to 3
    windows of a few hundred time units, so many lanes find no cut) with every window
    cut."""
    import test_oracle_pins as pins
    cut, _ = flags()
    for seed in range(120):
        net, stim = pins._random_case(seed)
        ref = oracle_lib.simulate(net, stim)
        assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), flags=cut), ref, "seed %d" % seed)


@pytest.mark.parametrize("case", ["busy", "slow", "zero"])
def test_cut_windows_hard_cases(gpu, oracle_lib, case):
    """busy: every input toggles every 60-unit cycle with glitch pairs, while a quiet
    time needs a gap of a whole gate delay (up to 60) plus twice the wire delay, so most
    searches give up and lanes take their neighbours' stretches; slow: gate delays of
    up to 5000 against 200-unit cycles, so no cut exists at all; zero: every delay 0
    (margins 0 and 1, zero-width output pulses)."""
    cut, _ = flags()
    if case == "busy":
        spec = synth.NetlistSpec(num_gates=2000, num_inputs=30, num_levels=8, seed=71, cond_fraction=0.4)
        st = synth.StimulusSpec(num_inputs=30, cycles=400, period=60, activity=1.0, windows=2, seed=71,
                                glitch_frac=0.5, glitch_span=(1, 4))
    elif case == "slow":
        spec = synth.NetlistSpec(num_gates=1500, num_inputs=24, num_levels=6, seed=72, gate_delay=(1000, 5000))
        st = synth.StimulusSpec(num_inputs=24, cycles=300, period=200, activity=0.5, windows=1, seed=72,
                                glitch_frac=0.2)
    else:
        spec = synth.NetlistSpec(num_gates=2000, num_inputs=30, num_levels=8, seed=73, gate_delay=(0, 0),
                                 wire_delay=(0, 0))
        st = synth.StimulusSpec(num_inputs=30, cycles=500, period=100, activity=0.5, windows=4, seed=73,
                                glitch_frac=0.3, glitch_span=(1, 3))
    net = synth.generate_netlist(spec)
    stim = synth.generate_stimulus(st)
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), flags=cut), ref, case)


def test_cut_windows_on_every_launch_path(gpu, oracle_lib):
    """Graph replay (twice), direct launches and timed launches, and packing to exact
    size, with cut windows."""
    from gate_level_logic_gb300 import gatspi
    cut, _ = flags()
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=2500, num_inputs=32, num_levels=10, seed=74,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=32, cycles=1500, period=400, activity=0.4,
                                                      windows=3, seed=74, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    pw = pool_for(ref, net)
    for extra in (0, gatspi.GATSPI_FLAG_NO_GRAPH, gatspi.GATSPI_FLAG_LEVEL_TIMING, gatspi.GATSPI_FLAG_COMPACT):
        assert_same(run_gpu(gpu, net, stim, pw, flags=cut | extra, repeat=2), ref, "flags %#x" % extra)


def test_load_switches_between_cut_and_whole_windows(gpu, oracle_lib):
    """One context of 4 windows: short windows (a few words per input) are simulated
    whole, long ones cut; each load that changes this re-captures the level graph, and
    every run equals the oracle."""
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=1200, num_inputs=20, num_levels=6, seed=75))
    short = synth.generate_stimulus(synth.StimulusSpec(num_inputs=20, cycles=400, period=100, activity=0.02,
                                                       windows=4, seed=75))
    long_ = synth.generate_stimulus(synth.StimulusSpec(num_inputs=20, cycles=400, period=100, activity=0.5,
                                                       windows=4, seed=76, glitch_frac=0.3))
    assert np.array_equal(short.window_len, long_.window_len)
    refs = {"short": oracle_lib.simulate(net, short), "long": oracle_lib.simulate(net, long_)}
    words = {"short": short.pi_words.size / (20 * 4), "long": long_.pi_words.size / (20 * 4)}
    assert words["short"] < 32 <= words["long"]
    pw = max(pool_for(r, net) for r in refs.values())
    with gpu(net, short.window_len, pool_words=pw) as sim:
        for name in ("short", "long", "long", "short", "long"):
            st = short if name == "short" else long_
            sim.load(st.pi_off, st.pi_words)
            assert sim.lanes_per_window() == (8 if name == "long" else 1)
            sim.simulate()
            tc, t0, t1 = sim.toggle_stats()
            off, pool = sim.export_all()
            assert_same(dict(off=off, pool=pool, tc=tc, t0=t0, t1=t1), refs[name], name)


def test_cut_windows_missing_arc_and_stalled_scan(gpu, oracle_lib):
    """A missing arc met inside a cut window reports GATSPI_EBADLUT; a stalled scan
    before a cut level gives up with GATSPI_ETIMEOUT (the level kernels after it read
    no waveform through the unwritten window index); the same contexts then simulate
    exactly."""
    from gate_level_logic_gb300 import GatspiError, gatspi
    cut, _ = flags()
    tt = np.array([0, 0, 1, 1], np.uint8)                       # output = first pin
    D = np.full((8, 2), INF, np.int32)
    D[0, :] = 5                                                 # first pin rise -> output rise
    net = single_gate(tt, 2, D)
    edges = [0] + list(range(50, 5000, 400)) + [EOW]           # the first fall needs the missing arc
    st = synth.from_waveforms([[edges], [[0, 70, EOW]]], 6000)
    with gpu(net, st.window_len, pool_words=1 << 16, flags=cut) as sim:
        sim.load(st.pi_off, st.pi_words)
        assert sim.lanes_per_window() == 32
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_EBADLUT"
        rise_only = synth.from_waveforms([[[0, 50, EOW]], [[0, 70, EOW]]], 6000)
        ref = oracle_lib.simulate(net, rise_only)
        sim.load(rise_only.pi_off, rise_only.pi_words)
        sim.simulate()
        tc, t0, t1 = sim.toggle_stats()
        assert np.array_equal(tc, ref.tc) and np.array_equal(t1, ref.t1)

    big = synth.generate_netlist(synth.NetlistSpec(num_gates=12000, num_inputs=64, num_levels=6, seed=77))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=64, cycles=400, period=300, activity=0.5,
                                                      windows=2, seed=77, glitch_frac=0.2))
    ref = oracle_lib.simulate(big, stim, threads=THREADS)
    with gpu(big, stim.window_len, pool_words=pool_for(ref, big), flags=cut) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        gatspi.gatspi_inject_scan_stall(sim.ctx, 2, 20_000_000)   # 2000 gates: two scan tiles
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_ETIMEOUT", str(e.value)
        sim.simulate()
        tc, t0, t1 = sim.toggle_stats()
        off, pool = sim.export_all()
        assert_same(dict(off=off, pool=pool, tc=tc, t0=t0, t1=t1), ref, "after the stall")


def test_cut_window_flags_exclude_each_other(gpu):
    from gate_level_logic_gb300 import GatspiError
    cut, whole = flags()
    net, stim = synth.make("tiny")
    with pytest.raises(GatspiError) as e:
        gpu(net, stim.window_len, pool_words=1 << 16, flags=cut | whole)
    assert e.value.name == "GATSPI_EINVAL"


def test_one_window_segments(gpu, oracle_lib):
    """One window: a gate whose work exceeds its level's share per resident warp takes
    up to 8 warps, one per segment of the window between two quiet times, and the last
    warp to finish moves the segments together.  A lone gate per level always takes all
    8; a few heavy gates among many light ones take several; replays and a second
    context must find every per-gate counter reset."""
    cut, _ = flags()
    tt = np.array([0, 1, 1, 0], np.uint8)                       # XOR2
    D = np.full((8, 2), 7, np.int32)
    one = single_gate(tt, 2, D, wire_rise=[1, 2], wire_fall=[2, 1])
    stim1 = synth.generate_stimulus(synth.StimulusSpec(num_inputs=2, cycles=3000, period=200, activity=0.7,
                                                       windows=1, seed=81, glitch_frac=0.3))
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=4000, num_inputs=16, num_levels=8, seed=82,
                                                   cond_fraction=0.3, fanout_mean=6.0))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=16, cycles=4000, period=300, activity=0.6,
                                                      windows=1, seed=82, glitch_frac=0.2))
    for nt, st in ((one, stim1), (net, stim)):
        ref = oracle_lib.simulate(nt, st, threads=THREADS)
        for fl in (cut, 0):
            assert_same(run_gpu(gpu, nt, st, pool_for(ref, nt), flags=fl, repeat=3), ref, "flags %d" % fl)


def test_one_window_segments_after_a_stalled_scan(gpu, oracle_lib):
    """A stalled scan stops a one-window run in the middle of a level whose heavy gates
    are split into segments; the next simulates of the same context (direct and from
    the graph) must be exact, so no segment counter may carry over."""
    from gate_level_logic_gb300 import GatspiError, gatspi
    cut, _ = flags()
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=9000, num_inputs=40, num_levels=6, seed=83,
                                                   fanout_mean=5.0))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=40, cycles=2000, period=300, activity=0.5,
                                                      windows=1, seed=83, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net), flags=cut) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        assert sim.lanes_per_window() == 32
        gatspi.gatspi_inject_scan_stall(sim.ctx, 3, 20_000_000)   # 1500 gates: two scan tiles
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_ETIMEOUT", str(e.value)
        for _ in range(2):
            sim.simulate()
            tc, t0, t1 = sim.toggle_stats()
            off, pool = sim.export_all()
            assert_same(dict(off=off, pool=pool, tc=tc, t0=t0, t1=t1), ref, "after the stall")


@pytest.mark.parametrize("W", [2, 3, 4, 16])
def test_long_windows_of_heavy_gates(gpu, oracle_lib, W):
    """Two to sixteen long windows (thousands of words per input window) cut into
    stretches: a lone gate, a netlist of many gates with heavy ones, with and without
    packing, against the oracle."""
    from gate_level_logic_gb300 import gatspi
    cut, _ = flags()
    tt = np.array([0, 1, 1, 0], np.uint8)                       # XOR2
    D = np.full((8, 2), 9, np.int32)
    one = single_gate(tt, 2, D, wire_rise=[2, 0], wire_fall=[1, 3])
    stim1 = synth.generate_stimulus(synth.StimulusSpec(num_inputs=2, cycles=4000 * W, period=200, activity=0.7,
                                                       windows=W, seed=90 + W, glitch_frac=0.3))
    ref1 = oracle_lib.simulate(one, stim1)
    assert_same(run_gpu(gpu, one, stim1, pool_for(ref1, one), flags=cut, repeat=2), ref1, "lone gate")
    if W == 4:
        net = synth.generate_netlist(synth.NetlistSpec(num_gates=4000, num_inputs=16, num_levels=8, seed=95,
                                                       cond_fraction=0.3, fanout_mean=6.0))
        stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=16, cycles=8000, period=300, activity=0.6,
                                                          windows=W, seed=95, glitch_frac=0.2))
        ref = oracle_lib.simulate(net, stim, threads=THREADS)
        for fl in (cut, 0, cut | gatspi.GATSPI_FLAG_COMPACT):
            assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), flags=fl, repeat=2), ref, "flags %#x" % fl)


@pytest.mark.parametrize("q", [60, 0])
@pytest.mark.parametrize("W", [1, 3, 16])
def test_cut_windows_below_pulse_percent_100(gpu, oracle_lib, W, q):
    """PATHPULSEPERCENT below 100 (0: transport delay), cut and whole: several output
    entries can be pending, and a cancel in a stretch can expose the entry in effect at
    its cut, which the lane before wrote; against the oracle at the same percentage."""
    cut, whole = flags()
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=3001, num_inputs=37, num_levels=9, seed=700 + W,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=37, cycles=2000, period=300, activity=0.3,
                                                      windows=W, seed=W + 40, glitch_frac=0.3))
    ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=q)
    pw = pool_for(ref, net)
    with gpu(net, stim.window_len, pool_words=pw, flags=cut, pulse_percent=q) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        assert sim.lanes_per_window() == 32 // W
    assert_same(run_gpu(gpu, net, stim, pw, flags=cut, pulse_percent=q), ref, "cut W=%d q=%d" % (W, q))
    assert_same(run_gpu(gpu, net, stim, pw, flags=whole, pulse_percent=q), ref, "whole W=%d q=%d" % (W, q))


def test_cut_windows_random_small_netlists_below_100(gpu, oracle_lib):
    """The 120 corner-heavy cases cut at PATHPULSEPERCENT = 50."""
    import test_oracle_pins as pins
    cut, _ = flags()
    for seed in range(120):
        net, stim = pins._random_case(seed)
        ref = oracle_lib.simulate(net, stim, pulse_percent=50)
        assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), flags=cut, pulse_percent=50), ref,
                    "seed %d" % seed)


def test_cut_windows_below_100_segments_and_launch_paths(gpu, oracle_lib):
    """One window split into segments at PATHPULSEPERCENT = 40 (replayed), and three
    windows at 30 on every launch path, packing included."""
    from gate_level_logic_gb300 import gatspi
    cut, _ = flags()
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=4000, num_inputs=16, num_levels=8, seed=82,
                                                   cond_fraction=0.3, fanout_mean=6.0))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=16, cycles=4000, period=300, activity=0.6,
                                                      windows=1, seed=82, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=40)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), flags=cut, repeat=3, pulse_percent=40), ref,
                "segments q=40")
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=2500, num_inputs=32, num_levels=10, seed=74,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=32, cycles=1500, period=400, activity=0.4,
                                                      windows=3, seed=74, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=30)
    pw = pool_for(ref, net)
    for extra in (0, gatspi.GATSPI_FLAG_NO_GRAPH, gatspi.GATSPI_FLAG_LEVEL_TIMING, gatspi.GATSPI_FLAG_COMPACT):
        assert_same(run_gpu(gpu, net, stim, pw, flags=cut | extra, repeat=2, pulse_percent=30), ref,
                    "q=30 flags %#x" % extra)
