"""Pins of the oracle's testbench restructuring (whole-testbench input waveforms cut
into cycle windows; GATSPI page, Sections 1, 4 and 5).

* the stimulus generator cuts the same seeded edges into windows by its own,
  vectorised route (edges binned by window, counts, value at each window start):
  both must give the same arrays for many specs;
* hand-worked cuts: transitions on a window boundary fold into the later window's
  initial value; transitions past the last window are dropped; windows without
  transitions; an initial 1;
* one window as long as the testbench is the identity;
* invariant at any size: the windows put back on the testbench's time axis give
  the original transitions (those before the end of the last window).
"""
import numpy as np
import pytest

from helpers import EOW
from synth.stimulus import StimulusSpec, generate_stimulus, generate_testbench


def _specs():
    rng = np.random.default_rng(7)
    for seed in range(60):
        cycles = int(rng.integers(1, 300))
        yield StimulusSpec(num_inputs=int(rng.integers(1, 40)), cycles=cycles, period=int(rng.integers(3, 2000)),
                           activity=float(rng.choice([0.0, 0.01, 0.2, 0.7, 1.0])),
                           windows=int(rng.integers(1, cycles + 1)), seed=seed,
                           glitch_frac=float(rng.choice([0.0, 0.3])), glitch_span=(1, int(rng.integers(1, 30))),
                           max_offset=int(rng.choice([0, 2, 50])))


def test_restructure_equals_generator_windows(oracle_lib):
    n = 0
    for spec in _specs():
        if spec.glitch_frac > 0 and spec.period < 4:
            continue
        tb = generate_testbench(spec)
        st = generate_stimulus(spec)
        off, words = oracle_lib.restructure(tb.off, tb.words, tb.window_len)
        assert np.array_equal(off, st.pi_off), spec
        assert np.array_equal(words, st.pi_words), spec
        n += 1
    assert n >= 50


def _cut(oracle_lib, wave, window_len):
    off, words = oracle_lib.restructure([0, len(wave)], np.asarray(wave, np.int32), window_len)
    return [words[off[k]:off[k + 1]].tolist() for k in range(len(window_len))]


def test_boundary_transitions_fold_into_the_later_window(oracle_lib):
    # windows [0, 10), [10, 20), [20, 30): the toggle at 10 sets window 1's initial
    # value (0 after toggles at 5 and 10); 27 lands at 7 in window 2; 30 is past the end
    got = _cut(oracle_lib, [0, 5, 10, 15, 27, 30, EOW], [10, 10, 10])
    assert got == [[0, 5, EOW], [0, 5, EOW], [-1, 0, 7, EOW]]


def test_initial_one_and_quiet_windows(oracle_lib):
    got = _cut(oracle_lib, [-1, 0, 25, EOW], [10, 10, 10])
    assert got == [[-1, 0, EOW], [-1, 0, EOW], [-1, 0, 5, EOW]]
    assert _cut(oracle_lib, [0, EOW], [3, 4]) == [[0, EOW], [0, EOW]]


def test_uneven_windows(oracle_lib):
    # starts 0, 7, 8, 20: toggles at 3 and 7 leave the value 0, the one at 7 folding
    # into window 1; window 2 starts at 0 and holds 9 -> 1 and 19 -> 11; the toggle at
    # 20 makes window 3 start at 1
    got = _cut(oracle_lib, [0, 3, 7, 9, 19, 20, EOW], [7, 1, 12, 5])
    assert got == [[0, 3, EOW], [0, EOW], [0, 1, 11, EOW], [-1, 0, EOW]]


def test_single_window_is_identity(oracle_lib):
    tb = generate_testbench(StimulusSpec(num_inputs=30, cycles=200, period=100, activity=0.4, windows=1, seed=3,
                                         glitch_frac=0.3))
    off, words = oracle_lib.restructure(tb.off, tb.words, tb.window_len)
    assert np.array_equal(off, tb.off) and np.array_equal(words, tb.words)


def _transitions(wave):
    wave = list(wave)
    head = 2 if wave[0] == -1 else 1
    return wave[0] == -1, wave[head:-1]


@pytest.mark.parametrize("seed", range(6))
def test_windows_put_back_give_the_testbench(oracle_lib, seed):
    """Randomly placed toggles (boundaries included), uneven windows shorter than the
    testbench: every window's transitions shifted by its start, plus a transition at
    a start where the initial value differs from the value the window before ended
    with, are the testbench's transitions before the end of the last window."""
    rng = np.random.default_rng(seed)
    P = 12
    starts = np.cumsum(rng.integers(1, 40, size=int(rng.integers(1, 30))))
    window_len = np.diff(np.concatenate(([0], starts)))
    total = int(starts[-1]) + 50
    waves = []
    for p in range(P):
        t = np.unique(rng.integers(1, total, size=int(rng.integers(0, 40))))
        if p % 3 == 0:   # toggles on every boundary too
            t = np.unique(np.concatenate([t, starts[:-1]]))
        init = int(rng.integers(0, 2))
        waves.append(([-1, 0] if init else [0]) + t.tolist() + [EOW])
    tb_off = np.concatenate(([0], np.cumsum([len(w) for w in waves])))
    off, words = oracle_lib.restructure(tb_off, np.concatenate(waves).astype(np.int32), window_len)
    W = len(window_len)
    wstart = np.concatenate(([0], starts[:-1]))
    for p in range(P):
        init, trans = _transitions(waves[p])
        back, value = [], init
        for w in range(W):
            k = p * W + w
            first, rel = _transitions(words[off[k]:off[k + 1]])
            if first != value:
                back.append(int(wstart[w]))
            back += [int(wstart[w]) + r for r in rel]
            value = first ^ (len(rel) & 1)
        assert back == [t for t in trans if t < starts[-1]], p


def test_malformed_testbench_is_rejected(oracle_lib):
    for bad in ([0, 5, 5, EOW], [1, 5, EOW], [0, 5, 3, EOW], [-1, 1, 5, EOW], [0, 0, EOW], [0, 5]):
        with pytest.raises(oracle_lib.OracleError):
            _cut(oracle_lib, bad, [10])
