"""Parity of the device-side testbench restructuring (gatspi_load_testbench) with the
oracle's cut, and of the simulation that follows it with the oracle's simulation of
the oracle-cut windows.  Bit-exact.
"""
import os

import numpy as np
import pytest

import synth
from helpers import EOW
from synth.stimulus import StimulusSpec, generate_testbench
from test_gpu_parity import assert_same, gpu, pool_for  # noqa: F401  (gpu is a fixture)

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


def _oracle_windows(oracle_lib, tb):
    off, words = oracle_lib.restructure(tb.off, tb.words, tb.window_len)
    return synth.Stimulus(num_inputs=tb.num_inputs, num_windows=tb.num_windows, window_len=tb.window_len,
                          window_cycles=tb.window_cycles, pi_off=off, pi_words=words, stats={})


def _run(Simulator, net, tb, pool_words, device=False, **kw):
    import torch
    with Simulator(net, tb.window_len, pool_words=pool_words, **kw) as sim:
        if device:
            sim.load_testbench(torch.from_numpy(tb.off).cuda(), torch.from_numpy(tb.words).cuda())
        else:
            sim.load_testbench(tb.off, tb.words)
        sim.simulate()
        tc, t0, t1 = sim.toggle_stats()
        off, words = sim.export_all()
        return dict(off=off, pool=words, tc=tc, t0=t0, t1=t1)


def _pool(ref, net, tb):
    return pool_for(ref, net) + 2 * tb.words.size + 3 * tb.num_windows * tb.num_inputs + 4096


@pytest.mark.parametrize("name", ["tiny", "50k"])
def test_workload_testbench(gpu, oracle_lib, name):
    net, _ = synth.make(name)
    tb = synth.testbench(name)
    stim = _oracle_windows(oracle_lib, tb)
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(_run(gpu, net, tb, _pool(ref, net, tb)), ref, name)


@pytest.mark.parametrize("W", [1, 5, 31, 32, 33, 70, 257])
def test_window_counts(gpu, oracle_lib, W):
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=1500, num_inputs=45, num_levels=7, seed=200 + W,
                                                   cond_fraction=0.3))
    tb = generate_testbench(StimulusSpec(num_inputs=45, cycles=max(W, 300), period=300, activity=0.3, windows=W,
                                         seed=W, glitch_frac=0.3))
    stim = _oracle_windows(oracle_lib, tb)
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    assert_same(_run(gpu, net, tb, _pool(ref, net, tb)), ref, "W=%d" % W)


def test_toggles_on_window_boundaries_from_device_memory(gpu, oracle_lib):
    """Uneven windows, toggles on every boundary and past the last window, initial 1s,
    inputs without toggles; the testbench passed as CUDA tensors."""
    rng = np.random.default_rng(5)
    window_len = rng.integers(1, 60, size=45)
    starts = np.concatenate(([0], np.cumsum(window_len)))
    total = int(starts[-1])
    P = 23
    waves = []
    for p in range(P):
        t = np.unique(rng.integers(1, total + 80, size=int(rng.integers(0, 70))))
        if p % 2 == 0:
            t = np.unique(np.concatenate([t, starts[1:]]))
        if p == 7:
            t = np.zeros(0, np.int64)
        waves.append(([-1, 0] if p % 3 == 0 else [0]) + t.tolist() + [EOW])
    off = np.concatenate(([0], np.cumsum([len(w) for w in waves]))).astype(np.int64)
    tb = synth.Testbench(num_inputs=P, num_windows=len(window_len), window_len=window_len.astype(np.int64),
                         window_cycles=np.zeros(len(window_len), np.int64), off=off,
                         words=np.concatenate(waves).astype(np.int32))
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=400, num_inputs=P, num_levels=5, seed=9,
                                                   cond_fraction=0.3))
    stim = _oracle_windows(oracle_lib, tb)
    ref = oracle_lib.simulate(net, stim)
    for device in (False, True):
        assert_same(_run(gpu, net, tb, _pool(ref, net, tb), device=device), ref, "device=%s" % device)


def test_pulse_percent_after_testbench(gpu, oracle_lib):
    net, _ = synth.make("50k")
    tb = synth.testbench("50k")
    stim = _oracle_windows(oracle_lib, tb)
    ref = oracle_lib.simulate(net, stim, threads=THREADS, pulse_percent=40)
    assert_same(_run(gpu, net, tb, _pool(ref, net, tb), pulse_percent=40), ref, "q=40")


def test_bench_workload_inputs_and_statistics(gpu, oracle_lib):
    """The 1M-gate bench workload loaded from its testbench: sampled input windows equal
    the generator's windows, and the statistics and sampled gate windows equal those
    of the regular load."""
    from gate_level_logic_gb300 import Simulator
    net, stim = synth.make("1M")
    tb = synth.testbench("1M")
    sel = np.array([0, 1, 31, 32, 100, 255], dtype=np.int32)
    P, n = net.num_inputs, len(sel)
    res = []
    for use_tb in (True, False):
        with Simulator(net, stim.window_len, pool_words=6 << 30) as sim:
            if use_tb:
                sim.load_testbench(tb.off, tb.words)
            else:
                sim.load(stim.pi_off, stim.pi_words)
            sim.simulate()
            off, words = sim.export_windows(sel)
            res.append((sim.toggle_stats(), off, words))
    want = synth.select_windows(stim, sel)
    off, words = res[0][1], res[0][2]
    assert np.array_equal(off[:P * n + 1], want.pi_off)
    assert np.array_equal(words[:off[P * n]], want.pi_words)
    for a, b in zip(res[0][0], res[1][0]):
        assert np.array_equal(a, b)
    assert np.array_equal(res[0][1], res[1][1]) and np.array_equal(res[0][2], res[1][2])


def test_errors(gpu, oracle_lib):
    from gate_level_logic_gb300 import GatspiError
    net, _ = synth.make("tiny")
    tb = synth.testbench("tiny")
    with gpu(net, tb.window_len, pool_words=1 << 20) as sim:
        bad = tb.words.copy()
        bad[tb.off[3] + 3] = bad[tb.off[3] + 2]            # repeated timestamp in input 3
        with pytest.raises(GatspiError) as e:
            sim.load_testbench(tb.off, bad)
        assert e.value.name == "GATSPI_EBADWAVE" and "input 3" in str(e.value)
        with pytest.raises(GatspiError) as e:
            sim.simulate()
        assert e.value.name == "GATSPI_ESTATE"
        off = tb.off.copy()
        off[-1] += 1
        with pytest.raises(GatspiError) as e:
            sim.load_testbench(off, tb.words)
        assert e.value.name == "GATSPI_EINVAL"
        sim.load_testbench(tb.off, tb.words)                # the context is still usable
        sim.simulate()
        stim = _oracle_windows(oracle_lib, tb)
        assert np.array_equal(sim.toggle_stats()[0], oracle_lib.simulate(net, stim).tc)
    with gpu(net, tb.window_len, pool_words=tb.words.size + 64) as sim:
        with pytest.raises(GatspiError) as e:
            sim.load_testbench(tb.off, tb.words)
        assert e.value.name == "GATSPI_EPOOL_OVERFLOW"
