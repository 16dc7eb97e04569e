"""Full-size parity of the CUDA path (through the C ABI) with the CPU oracle.

The 5M-gate workload, the scan-style 500k-gate run and all sixteen points of the
activity x windows sweep are too large to compare word by word in a test, so the
oracle's complete run of each (every gate in every window) is stored as per-level
digests by ``tests/golden/make_digests.py`` and the GPU run is reduced the same way:
every net's waveforms hashed in window order by ``gatspi_net_digests`` and TC/T1 of
every gate from ``gatspi_toggle_stats``, compared level by level (exact sums and
position-keyed mixes; ``tests/digests.py``).  A difference in any word of any
(net, window) waveform, or in any gate's TC, T0 or T1, fails.

Also here: the digest entry point against digests of the exported waveforms and of
the oracle's pool, a stalled scan that must give up with GATSPI_ETIMEOUT, and two
contexts of different window counts in one process.
"""
import json
import os

import numpy as np
import pytest

import digests
import synth

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "digests")
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


def _release_device_memory():
    import gc

    import torch
    gc.collect()
    torch.cuda.empty_cache()


def _pool_for_device(net, W):
    """Pool words: the free device memory less the context's own arrays and a margin."""
    import torch
    _release_device_memory()          # the previous workload's pool back to the driver
    free, _ = torch.cuda.mem_get_info()
    nets = net.num_inputs + net.num_gates
    widest = int(np.diff(net.level_offsets).max())
    own = 10 * nets * W + 2 * widest * W + 16 * net.num_gates + 8 * net.num_inputs * W
    return int((free - own - (6 << 30)) // 4) // 4 * 4


def test_net_digests_match_exports_and_oracle(gpu, oracle_lib):
    """gatspi_net_digests equals the same FNV-1a computed on the host from the exported
    waveforms and from the oracle's pool, on 16 windows and on one long window."""
    cases = [synth.make("50k")]
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=1500, num_inputs=24, num_levels=6, seed=503,
                                                   cond_fraction=0.3))
    cases.append((net, synth.generate_stimulus(synth.StimulusSpec(num_inputs=24, cycles=3000, period=300,
                                                                  activity=0.6, windows=1, seed=3))))
    for net, stim in cases:
        ref = oracle_lib.simulate(net, stim, threads=THREADS)
        W = stim.num_windows
        with gpu(net, stim.window_len, pool_words=4 * ref.pool.size + 4096) as sim:
            sim.load(stim.pi_off, stim.pi_words)
            inputs_only = sim.net_digests(0, net.num_inputs)
            sim.simulate()
            got, counts = sim.net_digests(with_words=True)
            off, words = sim.export_all()
            part = sim.net_digests(net.num_inputs + 7, 5)
        expect = digests.net_digests(ref.off, ref.pool, net.num_nets, W)
        assert np.array_equal(digests.net_digests(off, words, net.num_nets, W), expect)
        assert np.array_equal(got, expect)
        assert np.array_equal(counts, np.diff(ref.off).reshape(net.num_nets, W).sum(axis=1))
        assert np.array_equal(inputs_only, expect[:net.num_inputs])
        assert np.array_equal(part, expect[net.num_inputs + 7:net.num_inputs + 12])
        d = oracle_lib.digest(net, stim, threads=THREADS)
        assert np.array_equal(d.net_hash, expect)


def test_net_digests_argument_checks(gpu):
    from gate_level_logic_gb300 import GatspiError
    net, stim = synth.make("tiny")
    with gpu(net, stim.window_len, pool_words=1 << 16) as sim:
        with pytest.raises(GatspiError) as e:
            sim.net_digests(0, 4)
        assert e.value.name == "GATSPI_ESTATE"          # nothing loaded
        sim.load(stim.pi_off, stim.pi_words)
        with pytest.raises(GatspiError) as e:
            sim.net_digests()
        assert e.value.name == "GATSPI_ESTATE"          # gates not simulated yet
        with pytest.raises(GatspiError) as e:
            sim.net_digests(net.num_nets - 1, 2)
        assert e.value.name == "GATSPI_EINVAL"
        assert sim.net_digests(0, 0).size == 0


def _golden(name):
    path = os.path.join(GOLDEN, name + ".json")
    assert os.path.exists(path), "no stored oracle digests for %s: run tests/golden/make_digests.py" % name
    with open(path) as f:
        return json.load(f)


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(digests.large_workloads()))
def test_full_size_against_oracle_digests(gpu, name):
    rec = _golden(name)
    _, make = digests.large_workloads()[name]
    q = digests.pulse_percent(name)
    assert rec.get("pulse_percent", 100) == q
    net, stim = make()
    assert digests.inputs_sha256(net, stim) == rec["inputs_sha256"], \
        "the generator drew other inputs than the stored oracle run"
    W = stim.num_windows
    try:
        with gpu(net, stim.window_len, pool_words=_pool_for_device(net, W), pulse_percent=q) as sim:
            sim.load(stim.pi_off, stim.pi_words)
            sim.simulate()
            tc, t0, t1 = sim.toggle_stats()
            h, words = sim.net_digests(with_words=True)
    finally:
        _release_device_memory()      # the pool took most of the device: give it back for later tests
    assert np.array_equal(t0 + t1, np.full(net.num_gates, rec["window_time"]))
    assert digests.input_record(net.num_inputs, h, words) == rec["inputs"]
    got = digests.level_records(net.level_offsets, net.num_inputs, h, words, tc, t1)
    for lvl, (g, e) in enumerate(zip(got, rec["levels"])):
        assert g == e, "level %d differs from the oracle: %s vs %s" % (lvl, g, e)
    assert int(tc.sum()) == rec["events"] and int(words.sum()) == rec["words"]


def test_stalled_scan_times_out_and_context_recovers(gpu, oracle_lib):
    """A stalled output-region scan (its first tile never taken: the next tiles wait
    for a flag nothing sets) gives up after the limit with GATSPI_ETIMEOUT instead of
    hanging; the next simulate of the same context is exact."""
    from gate_level_logic_gb300 import GatspiError, gatspi
    tiny, tstim = synth.make("tiny")      # 50 gates per level: a single scan tile, nothing to stall
    with gpu(tiny, tstim.window_len, pool_words=1 << 16) as sim:
        with pytest.raises(GatspiError) as e:
            gatspi.gatspi_inject_scan_stall(sim.ctx, 1, 10_000)
        assert e.value.name == "GATSPI_EINVAL"
    net, stim = synth.make("50k")         # 2500 gates per level: three scan tiles
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    with gpu(net, stim.window_len, pool_words=4 * ref.pool.size + 4096) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        with pytest.raises(GatspiError) as e:
            gatspi.gatspi_inject_scan_stall(sim.ctx, net.num_levels, 10_000)
        assert e.value.name == "GATSPI_EINVAL"
        for level in (3, 0):
            gatspi.gatspi_inject_scan_stall(sim.ctx, level, 20_000_000)   # 20 ms
            sim.simulate()
            with pytest.raises(GatspiError) as e:
                sim.sync()
            assert e.value.name == "GATSPI_ETIMEOUT", str(e.value)
            assert "level %d" % level in str(e.value)
            sim.simulate()
            tc, t0, t1 = sim.toggle_stats()
            assert np.array_equal(tc, ref.tc) and np.array_equal(t1, ref.t1)
        off, words = sim.export_all()
        assert np.array_equal(off, ref.off) and np.array_equal(words, ref.pool)


def test_contexts_with_different_window_counts(gpu, oracle_lib):
    """Contexts of many and of few windows in one process: creating the second (and an
    allocation-free call of few windows) leaves the first one's planning kernel able to
    launch, on the direct, timed and graph paths."""
    import torch
    from gate_level_logic_gb300 import gatspi
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=600, num_inputs=16, num_levels=4, seed=9))
    big = synth.generate_stimulus(synth.StimulusSpec(num_inputs=16, cycles=4096, period=50, activity=0.3,
                                                     windows=4096, seed=9))
    small = synth.generate_stimulus(synth.StimulusSpec(num_inputs=16, cycles=64, period=50, activity=0.3,
                                                       windows=16, seed=9))
    ref_big = oracle_lib.simulate(net, big, threads=THREADS)
    ref_small = oracle_lib.simulate(net, small)
    a = gpu(net, big.window_len, pool_words=4 * ref_big.pool.size + 4096, flags=gatspi.GATSPI_FLAG_NO_GRAPH)
    b = gpu(net, small.window_len, pool_words=4 * ref_small.pool.size + 4096)
    try:
        a.load(big.pi_off, big.pi_words)
        b.load(small.pi_off, small.pi_words)
        b.simulate()
        for timed in (False, True):
            a.set_level_timing(timed)
            a.simulate()
            tc, _, t1 = a.toggle_stats()
            assert np.array_equal(tc, ref_big.tc) and np.array_equal(t1, ref_big.t1)
        tc, _, t1 = b.toggle_stats()
        assert np.array_equal(tc, ref_small.tc) and np.array_equal(t1, ref_small.t1)
    finally:
        a.close()
        b.close()
    torch.cuda.synchronize()
