"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Waveforms, window offsets and toggle statistics are integers: the bar is bit-exact
equality.  Small and medium cases compare the whole pool; the 1M-gate workload (the
configuration bench.py times) compares the whole pool too.  The 5M-gate, scan-style
and sweep workloads are compared in full against stored oracle digests
(test_gpu_digests.py).
"""
import os

import numpy as np
import pytest

import synth
from helpers import EOW, INF, permute_pin_weights, single_gate, uniform_delays

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


def run_gpu(Simulator, net, stim, pool_words, flags=0, repeat=1, pulse_percent=100):
    """Simulate; return every waveform gathered gap-free (CSR, net-major) + statistics."""
    with Simulator(net, stim.window_len, pool_words=pool_words, flags=flags, pulse_percent=pulse_percent) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        for _ in range(repeat):
            sim.simulate()
        tc, t0, t1 = sim.toggle_stats()
        off, words = sim.export_all()
        return dict(off=off, pool=words, tc=tc, t0=t0, t1=t1, pool_used=sim.pool_used())


def assert_same(got, ref, what=""):
    assert np.array_equal(got["off"], ref.off), "window offsets differ " + what
    if not np.array_equal(got["pool"], ref.pool):
        bad = np.nonzero(got["pool"] != ref.pool)[0][:5] if got["pool"].size == ref.pool.size else "size"
        raise AssertionError("waveforms differ %s at %s" % (what, bad))
    assert np.array_equal(got["tc"], ref.tc), "TC differs " + what
    assert np.array_equal(got["t1"], ref.t1), "T1 differs " + what
    assert np.array_equal(got["t0"], ref.t0), "T0 differs " + what


def pool_for(ref, net=None):
    """Pool words the output regions need: inputs plus, per gate and chunk, the sum of
    its pins' source spans plus 3 words per window (the kernel's upper bound)."""
    P, G, W = ref.num_inputs, len(ref.tc), ref.num_windows
    net_words = np.diff(ref.off).reshape(P + G, W).sum(axis=1)
    if net is None:
        return int(4 * ref.pool.size) + 4096
    inputs = int(net_words[:P].sum())
    return inputs + int(net_words[net.fanin_net].sum()) + 3 * G * W + 4096


def test_tiny_full(gpu, oracle_lib):
    net, stim = synth.make("tiny")
    ref = oracle_lib.simulate(net, stim)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref)


def test_50k_full(gpu, oracle_lib):
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref)


@pytest.mark.parametrize("flags", [2])
def test_50k_launch_variants(gpu, oracle_lib, flags):
    """The level sequence launched directly instead of replayed from a graph."""
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), flags=flags), ref, "flags=%d" % flags)


@pytest.mark.parametrize("W", [1, 2, 3, 7, 16, 31, 32, 33, 63, 64, 65, 100, 128, 200, 256, 257, 384, 1024, 1025,
                               1500])
def test_window_counts(gpu, oracle_lib, W):
    """Ragged window chunks, several gates per warp (W < 32), ragged tiles, whole
    blocks of one gate's chunks (W = 128, 256, 384), the most windows that are ranked
    (1024) and windows taken in window order beyond it (1025, 1500)."""
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=3001, num_inputs=37, num_levels=9, seed=W,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=37, cycles=max(W, 300), period=500,
                                                      activity=0.2, windows=W, seed=W, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref, "W=%d" % W)


@pytest.mark.parametrize("W", [1, 3, 6])
def test_long_windows(gpu, oracle_lib, W):
    """Windows of hundreds to thousands of words: lengths of 255 and more, which the
    planner reads exactly from the window index instead of the one-byte lengths."""
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=1500, num_inputs=24, num_levels=6, seed=500 + W,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=24, cycles=3000, period=300, activity=0.6,
                                                      windows=W, seed=W, glitch_frac=0.2))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    lens = np.diff(ref.off)
    assert lens.max() > 700 and (lens >= 255).mean() > 0.2
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref, "W=%d" % W)


def test_long_windows_in_window_order(gpu, oracle_lib):
    """More than 1024 windows (taken in window order) of 255 words and more: the
    planner reads those lengths exactly from the window index."""
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=300, num_inputs=24, num_levels=4, seed=611,
                                                   cond_fraction=0.3))
    W = 1025
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=24, cycles=W * 260, period=300, activity=1.0,
                                                      windows=W, seed=11))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    lens = np.diff(ref.off)
    assert (lens >= 255).mean() > 0.5
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref, "W=%d" % W)


def test_random_small_netlists(gpu, oracle_lib):
    """The seeded corner-heavy cases the oracle was pinned on (zero delays, zero-width
    pulses, 1-4 pin random cells, conditional arcs, multiple windows)."""
    import test_oracle_pins as pins
    for seed in range(120):
        net, stim = pins._random_case(seed)
        ref = oracle_lib.simulate(net, stim)
        assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref,
                    "seed %d" % seed)


def test_permuted_pin_weights(gpu, oracle_lib):
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=2000, num_inputs=40, num_levels=8, seed=21,
                                                   cond_fraction=0.4))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=40, cycles=200, period=300, activity=0.3,
                                                      windows=40, seed=21, glitch_frac=0.2))
    perm = permute_pin_weights(net, seed=21)
    ref = oracle_lib.simulate(perm, stim, threads=THREADS)
    assert_same(run_gpu(gpu, perm, stim, pool_for(ref, perm)), ref, "permuted weights")
    assert np.array_equal(ref.pool, oracle_lib.simulate(net, stim, threads=THREADS).pool)


def test_simultaneous_switching_of_all_pins(gpu, oracle_lib):
    """Every pin of a gate driven by one source with equal wire delays: 2, 3 and 4
    pins switch at the same instant (the smallest-arc rule and the pin advance of
    every switching pin)."""
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=3000, num_inputs=32, num_levels=10, seed=31,
                                                   cond_fraction=0.5))
    fo = net.fanin_off
    first = np.repeat(net.fanin_net[fo[:-1]], np.diff(fo))
    rise = np.repeat(net.wire_rise[fo[:-1]], np.diff(fo))
    fall = np.repeat(net.wire_fall[fo[:-1]], np.diff(fo))
    net.fanin_net, net.wire_rise, net.wire_fall = first.astype(np.int32), rise, fall
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=32, cycles=300, period=200, activity=0.4,
                                                      windows=50, seed=31, glitch_frac=0.3, glitch_span=(1, 5)))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref)


def test_quiet_inputs_and_empty_level(gpu, oracle_lib):
    tts = [synth.truth_table("NAND2"), synth.truth_table("INV")]
    D2 = uniform_delays(2, 3, 4, tts[0])
    D1 = uniform_delays(1, 2, 2, tts[1])
    net = synth.build_netlist(num_inputs=2, level_gates=[2, 0, 1], type_names=["NAND2", "INV"],
                              type_num_pins=[2, 1], type_tts=tts, gate_type=[0, 1, 0],
                              fanins=[[0, 1], [0], [2, 3]], wire_rise=np.zeros(5), wire_fall=np.ones(5),
                              delay_tables=[D2, D1, D2])
    for waves in ([[0, EOW], [-1, 0, EOW]], [[0, 5, 9, 40, EOW], [-1, 0, 20, EOW]]):
        stim = synth.from_waveforms([[w] for w in waves], 100)
        ref = oracle_lib.simulate(net, stim)
        assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref)


def test_maximum_activity(gpu, oracle_lib):
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=4000, num_inputs=64, num_levels=16, seed=5,
                                                   cond_fraction=0.5))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=64, cycles=256, period=200, activity=1.0,
                                                      windows=64, seed=5, glitch_frac=0.5, glitch_span=(1, 4)))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref)


def test_level_timing_switch(gpu, oracle_lib):
    """Per-level times exist only after a timed run; switching timing on and off
    between runs of one context changes nothing in the results."""
    from gate_level_logic_gb300 import GatspiError
    net, stim = synth.make("tiny")
    ref = oracle_lib.simulate(net, stim)
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.level_times()
        assert e.value.name == "GATSPI_ESTATE"
        sim.set_level_timing(True)
        sim.simulate()
        lt, bt = sim.level_times()
        assert lt.shape == (net.num_levels,) and (lt > 0).all() and (bt > 0).all()
        sim.set_level_timing(False)
        sim.simulate()
        tc, t0, t1 = sim.toggle_stats()
        assert np.array_equal(tc, ref.tc) and np.array_equal(t1, ref.t1)


def test_toggle_stats_view(gpu, oracle_lib):
    """The zero-copy statistics equal the copied ones and the oracle's."""
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        tc, t1, ws = sim.toggle_stats_view()
        ctc, ct0, ct1 = sim.toggle_stats()
        assert not tc.flags.writeable
        assert np.array_equal(tc.astype(np.int64), ref.tc) and np.array_equal(t1.astype(np.int64), ref.t1)
        assert np.array_equal(ctc, ref.tc) and np.array_equal(ws - t1.astype(np.int64), ct0)


def test_replay_is_deterministic(gpu, oracle_lib):
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), repeat=3), ref, "after 3 replays")


def test_errors_leave_context_usable(gpu, oracle_lib):
    from gate_level_logic_gb300 import GatspiError
    net, stim = synth.make("tiny")
    ref = oracle_lib.simulate(net, stim)
    # pool too small for the outputs: reported at the next synchronising call; a quiet
    # stimulus needs regions of 3 words per gate and window and fits
    small = int(stim.pi_words.size) + 3 * net.num_gates + 64
    assert small < ref.pool.size
    with gpu(net, stim.window_len, pool_words=small) as sim:
        with pytest.raises(GatspiError) as e:
            sim.simulate()
        assert e.value.name == "GATSPI_ESTATE"
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.toggle_stats()
        assert e.value.name == "GATSPI_EPOOL_OVERFLOW"
        # a quiet stimulus fits: the same context simulates correctly afterwards
        quiet = synth.from_waveforms([[[0, EOW]] for _ in range(net.num_inputs)], stim.window_len)
        sim.load(quiet.pi_off, quiet.pi_words)
        sim.simulate()
        tc, _, _ = sim.toggle_stats()
        assert (tc == 0).all()
    # malformed input waveforms are rejected at load
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        bad = stim.pi_words.copy()
        bad[stim.pi_off[3] + 2] = bad[stim.pi_off[3] + 1]       # repeated timestamp
        with pytest.raises(GatspiError) as e:
            sim.load(stim.pi_off, bad)
        assert e.value.name == "GATSPI_EBADWAVE"
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        tc, _, _ = sim.toggle_stats()
        assert np.array_equal(tc, ref.tc)
    # an output change whose switching arcs are all missing
    tt = np.array([0, 0, 1, 1], np.uint8)
    lut = single_gate(tt, 2, np.full((8, 2), INF, np.int32))
    st = synth.from_waveforms([[[0, 50, EOW]], [[0, EOW]]], 100)
    with gpu(lut, st.window_len, pool_words=1024) as sim:
        sim.load(st.pi_off, st.pi_words)
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_EBADLUT"


@pytest.mark.parametrize("q", [100, 50, 0])
def test_missing_arc_after_valid_events(gpu, oracle_lib, q):
    """A buffer whose output-fall arc is missing: the rise at 50 is simulated, the
    fall at 120 meets the missing arc and the run reports GATSPI_EBADLUT at every
    PATHPULSEPERCENT; the same context then simulates a stimulus that never needs
    the arc, and the oracle agrees on it."""
    from gate_level_logic_gb300 import GatspiError
    tt = np.array([0, 0, 1, 1], np.uint8)                       # output = first pin
    D = np.full((8, 2), INF, np.int32)
    D[0, :] = 5                                                 # first pin rise -> output rise
    net = single_gate(tt, 2, D)
    st = synth.from_waveforms([[[0, 50, 120, 300, EOW]], [[0, 70, EOW]]], 400)
    with gpu(net, st.window_len, pool_words=4096, pulse_percent=q) as sim:
        sim.load(st.pi_off, st.pi_words)
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_EBADLUT"
        rise_only = synth.from_waveforms([[[0, 50, EOW]], [[0, 70, EOW]]], 400)
        ref = oracle_lib.simulate(net, rise_only, pulse_percent=q)
        sim.load(rise_only.pi_off, rise_only.pi_words)
        sim.simulate()
        tc, t0, t1 = sim.toggle_stats()
        assert np.array_equal(tc, ref.tc) and np.array_equal(t1, ref.t1)


def test_single_waveform_and_window_export(gpu, oracle_lib):
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        for net_id, w in [(0, 0), (255, 15), (256, 3), (net.num_inputs + net.num_gates - 1, 15), (30000, 7)]:
            assert np.array_equal(sim.waveform(net_id, w), ref.wave(net_id, w))
        sel = [15, 0, 7, 7]
        off, words = sim.export_windows(sel)
        sub = oracle_lib.simulate(net, synth.select_windows(stim, sel))
        assert np.array_equal(off, sub.off) and np.array_equal(words, sub.pool)


@pytest.mark.slow
def test_1M_full(gpu, oracle_lib):
    """The configuration bench.py times: 1M gates, 40 levels, 256 windows; whole pool,
    also with every level packed to its exact size (GATSPI_FLAG_COMPACT)."""
    from gate_level_logic_gb300 import gatspi
    net, stim = synth.make("1M")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref, "1M")
    got = run_gpu(gpu, net, stim, pool_for(ref, net), flags=gatspi.GATSPI_FLAG_COMPACT, repeat=2)
    assert_same(got, ref, "1M packed")
    assert got["pool_used"] <= 1.3 * ref.pool.size


@pytest.mark.parametrize("W", [1, 3, 16, 33, 256, 1025])
@pytest.mark.parametrize("q", [100, 40])
def test_compact_levels(gpu, oracle_lib, W, q):
    """Every level packed to its exact size after it is simulated: the same waveforms
    and statistics, the pool holding the waveforms plus one level's bound-sized
    regions; two runs in a row (the packing rewrites the window index)."""
    from gate_level_logic_gb300 import gatspi
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=2600, num_inputs=31, num_levels=7, seed=700 + W,
                                                   cond_fraction=0.3))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=31, cycles=max(W, 300), period=400,
                                                      activity=0.3, windows=W, seed=W, glitch_frac=0.3))
    ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=q)
    got = run_gpu(gpu, net, stim, pool_for(ref, net), flags=gatspi.GATSPI_FLAG_COMPACT, repeat=2, pulse_percent=q)
    assert_same(got, ref, "packed W=%d q=%d" % (W, q))
    # the packed waveforms plus at most one level's bound-sized regions
    P, G = net.num_inputs, net.num_gates
    words = np.diff(ref.off).reshape(P + G, W).sum(axis=1)
    lo = np.asarray(net.level_offsets)
    level_bound = max(int(words[net.fanin_net[net.fanin_off[a]:net.fanin_off[b]]].sum()) + 3 * (b - a) * W
                      for a, b in zip(lo[:-1], lo[1:]))
    assert ref.pool.size <= got["pool_used"] <= ref.pool.size + level_bound


def test_compact_pool_too_small(gpu, oracle_lib):
    """A pool with room for the waveforms but not for a level's bound-sized regions
    on top of the packed front: GATSPI_EPOOL_OVERFLOW, and the context still works
    with a quiet stimulus."""
    from gate_level_logic_gb300 import GatspiError, gatspi
    net, stim = synth.make("tiny")
    ref = oracle_lib.simulate(net, stim)
    with gpu(net, stim.window_len, pool_words=int(ref.pool.size * 1.02) // 4 * 4 + 4,
             flags=gatspi.GATSPI_FLAG_COMPACT) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_EPOOL_OVERFLOW"
        quiet = synth.from_waveforms([[[0, EOW]] for _ in range(net.num_inputs)], stim.window_len)
        sim.load(quiet.pi_off, quiet.pi_words)
        sim.simulate()
        tc, _, _ = sim.toggle_stats()
        assert (tc == 0).all()


# ---- PATHPULSEPERCENT below 100 (several pending output events; transport at 0) ----

@pytest.mark.parametrize("q", [0, 35, 70, 99])
def test_pulse_percent_random_small(gpu, oracle_lib, q):
    """The seeded corner-heavy cases at other pulse limits (a cancel re-reads the
    exposed entry from the lane's own output)."""
    import test_oracle_pins as pins
    for seed in range(40):
        net, stim = pins._random_case(seed)
        ref = oracle_lib.simulate(net, stim, pulse_percent=q)
        assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), pulse_percent=q), ref, "q=%d seed %d" % (q, seed))


@pytest.mark.parametrize("q", [0, 50, 80])
def test_pulse_percent_50k(gpu, oracle_lib, q):
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=q)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), pulse_percent=q), ref, "q=%d" % q)
    if q == 0:     # transport delay lets every pulse through: more toggles than the inertial default
        assert ref.tc.sum() > oracle_lib.simulate(net, stim, threads=THREADS).tc.sum()


@pytest.mark.parametrize("W", [5, 32, 70, 128])
def test_pulse_percent_window_counts(gpu, oracle_lib, W):
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=2500, num_inputs=29, num_levels=8, seed=100 + W,
                                                   cond_fraction=0.4))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=29, cycles=max(W, 200), period=400,
                                                      activity=0.3, windows=W, seed=W, glitch_frac=0.4))
    for q in (10, 60):
        ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=q)
        assert_same(run_gpu(gpu, net, stim, pool_for(ref, net), pulse_percent=q), ref,
                    "q=%d W=%d" % (q, W))


@pytest.mark.parametrize("seed", [77, 78])
def test_many_windows(gpu, oracle_lib, seed):
    """256 windows (eight groups of ranks per gate), high activity."""
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=1200, num_inputs=33, num_levels=6, seed=seed,
                                                   cond_fraction=0.5))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=33, cycles=512, period=400, activity=0.5,
                                                      windows=256, seed=seed, glitch_frac=0.4))
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref, "seed %d" % seed)


def test_empty_level_and_errors_many_windows(gpu, oracle_lib):
    """An empty level with 128 windows, then a missing delay arc reported with the
    context still usable."""
    from gate_level_logic_gb300 import GatspiError
    tt = synth.truth_table("NAND2")
    D = uniform_delays(2, 5, 7, tt)
    net = synth.build_netlist(num_inputs=2, level_gates=[1, 0, 1], type_names=["NAND2"], type_num_pins=[2],
                              type_tts=[tt], gate_type=[0, 0], fanins=[[0, 1], [2, 1]], wire_rise=np.zeros(4),
                              wire_fall=np.zeros(4), delay_tables=[D, D])
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=2, cycles=256, period=50, activity=0.5,
                                                      windows=128, seed=3))
    ref = oracle_lib.simulate(net, stim)
    assert_same(run_gpu(gpu, net, stim, pool_for(ref, net)), ref, "empty level")
    bad = np.full_like(D, INF)
    net2 = synth.build_netlist(num_inputs=2, level_gates=[1, 0, 1], type_names=["NAND2"], type_num_pins=[2],
                               type_tts=[tt], gate_type=[0, 0], fanins=[[0, 1], [2, 1]], wire_rise=np.zeros(4),
                               wire_fall=np.zeros(4), delay_tables=[D, bad])
    with gpu(net2, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        with pytest.raises(GatspiError) as e:
            sim.sync()
        assert e.value.name == "GATSPI_EBADLUT"
        sim.simulate()      # the context is still usable
        with pytest.raises(GatspiError):
            sim.sync()
