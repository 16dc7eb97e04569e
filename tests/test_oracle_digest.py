"""Pins of the oracle's digest driver (oracle.digest) and of the digest helpers.

The digest driver runs the same per-task routine as oracle.simulate with a
level-parallel schedule and keeps no merged pool; it is pinned to oracle.simulate
(itself pinned by brute force, goldens and mutations) by hashing the latter's
whole pool, for several thread counts, window batches and PATHPULSEPERCENT values.
The hash is pinned to the published FNV-1a 64 test vectors.
"""
import numpy as np
import pytest

import digests
import synth


# 64-bit FNV-1a of "", "a" and "foobar" (the FNV reference test vectors)
FNV_VECTORS = [(b"", 0xCBF29CE484222325), (b"a", 0xAF63DC4C8601EC8C), (b"foobar", 0x85944171F73967E8)]


@pytest.mark.parametrize("data,want", FNV_VECTORS)
def test_fnv1a64_vectors(oracle_lib, data, want):
    assert oracle_lib.fnv1a64(data) == want
    assert digests.fnv1a64(data) == want


def test_net_digests_helper_is_fnv_of_the_concatenated_windows():
    rng = np.random.default_rng(0)
    nets, W = 7, 3
    lens = rng.integers(2, 9, size=nets * W)
    off = np.concatenate(([0], np.cumsum(lens)))
    words = rng.integers(-2**31, 2**31 - 1, size=int(off[-1]), dtype=np.int64).astype(np.int32)
    got = digests.net_digests(off, words, nets, W)
    for n in range(nets):
        raw = words[off[n * W]:off[(n + 1) * W]].astype("<i4").tobytes()
        assert int(got[n]) == digests.fnv1a64(raw)


def _cases():
    yield "tiny", synth.make("tiny")
    yield "50k", synth.make("50k")
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=1500, num_inputs=24, num_levels=6, seed=503,
                                                   cond_fraction=0.3))
    yield "long", (net, synth.generate_stimulus(synth.StimulusSpec(num_inputs=24, cycles=3000, period=300,
                                                                   activity=0.6, windows=3, seed=3,
                                                                   glitch_frac=0.2)))


@pytest.mark.parametrize("q", [100, 40])
def test_digest_driver_equals_simulate(oracle_lib, q):
    for name, (net, stim) in _cases():
        ref = oracle_lib.simulate(net, stim, threads=4, pulse_percent=q)
        want = digests.net_digests(ref.off, ref.pool, net.num_nets, stim.num_windows)
        words = np.diff(ref.off).reshape(net.num_nets, stim.num_windows).sum(axis=1)
        for threads in (1, 3, 8):
            d = oracle_lib.digest(net, stim, threads=threads, pulse_percent=q)
            assert np.array_equal(d.net_hash, want), (name, threads)
            assert np.array_equal(d.net_words, words), (name, threads)
            assert np.array_equal(d.tc, ref.tc) and np.array_equal(d.t1, ref.t1), (name, threads)
            assert d.window_time == int(stim.window_len.sum())


def test_digest_in_window_batches():
    import oracle
    net, stim = synth.make("50k")
    whole = oracle.digest(net, stim, threads=4)
    state = None
    for a, b in [(0, 1), (1, 9), (9, 16)]:
        state = oracle.digest(net, synth.select_windows(stim, np.arange(a, b)), state=state, threads=2)
    assert np.array_equal(state.net_hash, whole.net_hash)
    assert np.array_equal(state.tc, whole.tc) and np.array_equal(state.t1, whole.t1)
    # out of order the digests differ (the hash follows window order), the sums do not
    state = None
    for a, b in [(9, 16), (0, 9)]:
        state = oracle.digest(net, synth.select_windows(stim, np.arange(a, b)), state=state, threads=2)
    assert not np.array_equal(state.net_hash, whole.net_hash)
    assert np.array_equal(state.tc, whole.tc)


def test_level_records_see_every_change():
    """A one-bit change of one gate's digest, TC or T1, or two gates trading values,
    changes that level's record."""
    rng = np.random.default_rng(1)
    P, G = 5, 40
    lo = np.array([0, 10, 25, 40])
    h = rng.integers(0, 2**63, size=P + G, dtype=np.int64).view(np.uint64)
    nw = rng.integers(2, 50, size=P + G)
    tc = rng.integers(0, 100, size=G)
    t1 = rng.integers(0, 10**6, size=G)
    base = digests.level_records(lo, P, h, nw, tc, t1)
    for arr, i in [(h, P + 12), (tc, 30), (t1, 3)]:
        mod = arr.copy()
        mod[i] ^= 1
        args = [h, nw, tc, t1]
        args[[id(h), id(nw), id(tc), id(t1)].index(id(arr))] = mod
        assert digests.level_records(lo, P, *args) != base
    swapped = tc.copy()
    swapped[[11, 12]] = swapped[[12, 11]]
    if tc[11] != tc[12]:
        assert digests.level_records(lo, P, h, nw, swapped, t1)[1]["tc_mix"] != base[1]["tc_mix"]
