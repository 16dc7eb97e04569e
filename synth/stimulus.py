"""Seeded primary-input stimulus, cut into independent cycle windows.

Waveform format (GATSPI page, Fig. 3): an int32 array of toggle timestamps whose
index parity is the logic value (even index = 0, odd index = 1).  A waveform that
starts at 1 begins with -1, 0 so that time 0 sits at an odd index; one that starts
at 0 begins with 0.  The array ends with EOW = INT32_MAX.

Every window is an independent re-simulation (cycle parallelism): its timestamps
are relative to the window start and each input starts at its value at that
instant.  Windows hold floor(C/W) or ceil(C/W) cycles, the first C mod W windows
taking the extra cycle.

Stimulus readings: initial input values are Bernoulli(0.5); in each cycle an input
toggles with probability ``activity`` at a uniform offset in [1, period-1]; with
probability ``glitch_frac`` a toggle is issued as a glitch pair whose second edge
follows the first by U{glitch_span} time units, clipped to the cycle.

The output is a CSR array pair: ``pi_off`` (int64, (P*W)+1 entries, net-major,
window-minor) and ``pi_words`` (int32).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

EOW = np.int32(2**31 - 1)


@dataclass
class StimulusSpec:
    num_inputs: int
    cycles: int
    period: int
    activity: float
    windows: int
    seed: int
    glitch_frac: float = 0.0
    glitch_span: tuple = (1, 20)
    max_offset: int = 0          # 0: toggles anywhere in [1, period-1]; else in [1, max_offset]


@dataclass
class Stimulus:
    num_inputs: int
    num_windows: int
    window_len: np.ndarray   # int64 [W], time units
    window_cycles: np.ndarray  # int64 [W]
    pi_off: np.ndarray       # int64 [P*W + 1]
    pi_words: np.ndarray     # int32
    stats: dict

    def window(self, pi: int, w: int) -> np.ndarray:
        k = pi * self.num_windows + w
        return self.pi_words[self.pi_off[k]:self.pi_off[k + 1]]


def window_cycles(cycles: int, windows: int) -> np.ndarray:
    base, extra = divmod(cycles, windows)
    wc = np.full(windows, base, dtype=np.int64)
    wc[:extra] += 1
    return wc


def _draw_edges(spec: StimulusSpec):
    """The seeded input edges: initial values and (input, cycle, offset) of every edge,
    sorted by input, then time."""
    rng = np.random.default_rng(spec.seed)
    P, C, T, W = spec.num_inputs, spec.cycles, spec.period, spec.windows
    if W < 1 or W > C:
        raise ValueError("need 1 <= windows <= cycles")
    if T < 3:
        raise ValueError("period must be >= 3")
    init = rng.integers(0, 2, size=P, dtype=np.int64)

    # toggle cycles per input: geometric gaps, drawn in one block with a safe margin
    p = float(spec.activity)
    if p > 0:
        mean = C * p
        M = int(mean + 8 * np.sqrt(mean + 1) + 16)
        gaps = rng.geometric(p, size=(P, M)) if p < 1 else np.ones((P, M), dtype=np.int64)
        cyc = np.cumsum(gaps, axis=1) - 1                       # 0-based cycle index
        keep = cyc < C
        if keep[:, -1].any():
            raise RuntimeError("stimulus margin too small")
        pi_of = np.broadcast_to(np.arange(P)[:, None], cyc.shape)[keep]
        cyc = cyc[keep]
    else:
        pi_of = np.zeros(0, dtype=np.int64)
        cyc = np.zeros(0, dtype=np.int64)
    n_tog = cyc.size
    glitch = rng.random(n_tog) < spec.glitch_frac
    top = T - 1 if spec.max_offset <= 0 else min(int(spec.max_offset), T - 1)
    if top < 2 and spec.glitch_frac > 0:
        raise ValueError("glitch pairs need room for two edges in a cycle")
    off1 = np.where(glitch, rng.integers(1, max(top, 2), size=n_tog), rng.integers(1, top + 1, size=n_tog))
    gl_lo, gl_hi = spec.glitch_span
    off2 = np.minimum(off1 + rng.integers(gl_lo, gl_hi + 1, size=n_tog), top)

    # edges: (pi, absolute time); glitch pairs contribute two edges
    e_pi = np.concatenate([pi_of, pi_of[glitch]])
    e_cyc = np.concatenate([cyc, cyc[glitch]])
    e_off = np.concatenate([off1, off2[glitch]])
    order = np.lexsort((e_off, e_cyc, e_pi))
    return init, e_pi[order], e_cyc[order], e_off[order], n_tog, int(glitch.sum())


def generate_stimulus(spec: StimulusSpec) -> Stimulus:
    P, C, T, W = spec.num_inputs, spec.cycles, spec.period, spec.windows
    init, e_pi, e_cyc, e_off, n_tog, n_glitch = _draw_edges(spec)

    wc = window_cycles(C, W)
    wstart = np.concatenate(([0], np.cumsum(wc)))          # first cycle of each window
    e_win = np.searchsorted(wstart, e_cyc, side="right") - 1
    e_rel = (e_cyc - wstart[e_win]) * T + e_off              # window-relative time

    # per (pi, window): edge counts and the value at the window start
    key = e_pi * W + e_win
    cnt = np.bincount(key, minlength=P * W).reshape(P, W)
    before = np.zeros((P, W), dtype=np.int64)
    before[:, 1:] = np.cumsum(cnt, axis=1)[:, :-1]
    v0 = (init[:, None] + before) & 1                       # value at the window start
    head = 1 + v0                                            # [0] or [-1, 0]
    length = head + cnt + 1
    pi_off = np.zeros(P * W + 1, dtype=np.int64)
    pi_off[1:] = np.cumsum(length.ravel())
    words = np.empty(int(pi_off[-1]), dtype=np.int32)
    starts = pi_off[:-1].reshape(P, W)
    # head words
    s1 = starts[v0 == 1]
    words[s1] = -1
    words[s1 + 1] = 0
    words[starts[v0 == 0]] = 0
    # edges: position = start + head + rank within (pi, window)
    first_edge = np.zeros(P * W + 1, dtype=np.int64)
    first_edge[1:] = np.cumsum(cnt.ravel())
    rank = np.arange(key.size) - first_edge[key]
    words[(starts.ravel() + head.ravel())[key] + rank] = e_rel.astype(np.int32)
    words[pi_off[1:] - 1] = EOW

    stats = {
        "toggles": int(n_tog),
        "glitch_pairs": n_glitch,
        "edges": int(e_pi.size),
        "words": int(words.size),
    }
    return Stimulus(num_inputs=P, num_windows=W, window_len=wc * T, window_cycles=wc,
                    pi_off=pi_off, pi_words=words, stats=stats)


def select_windows(stim: Stimulus, windows) -> Stimulus:
    """The stimulus of a subset of windows (windows are independent simulations)."""
    windows = np.asarray(windows, dtype=np.int64)
    P, W = stim.num_inputs, stim.num_windows
    k = (np.arange(P)[:, None] * W + windows[None, :]).ravel()
    lens = stim.pi_off[k + 1] - stim.pi_off[k]
    off = np.zeros(k.size + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens)
    src = np.repeat(stim.pi_off[k], lens) + (np.arange(int(off[-1])) - np.repeat(off[:-1], lens))
    return Stimulus(num_inputs=P, num_windows=len(windows), window_len=stim.window_len[windows],
                    window_cycles=stim.window_cycles[windows], pi_off=off,
                    pi_words=stim.pi_words[src], stats=dict(stim.stats))


def from_waveforms(waves, window_len) -> Stimulus:
    """Build a stimulus from explicit per-(pi, window) arrays: ``waves[pi][w]``."""
    P = len(waves)
    W = len(waves[0])
    flat = [np.asarray(waves[p][w], dtype=np.int32) for p in range(P) for w in range(W)]
    off = np.zeros(P * W + 1, dtype=np.int64)
    off[1:] = np.cumsum([a.size for a in flat])
    wl = np.asarray(window_len, dtype=np.int64).reshape(-1)
    if wl.size == 1:
        wl = np.repeat(wl, W)
    return Stimulus(num_inputs=P, num_windows=W, window_len=wl, window_cycles=np.zeros(W, dtype=np.int64),
                    pi_off=off, pi_words=np.concatenate(flat) if flat else np.zeros(0, np.int32), stats={})


@dataclass
class Testbench:
    """Whole-testbench input waveforms, before the cut into cycle windows: one Fig. 3
    array per input with times from the start of the testbench, and the lengths of
    the windows it is to be cut into (window w starts at the sum of the lengths of
    the windows before it)."""
    num_inputs: int
    num_windows: int
    window_len: np.ndarray     # int64 [W]
    window_cycles: np.ndarray  # int64 [W]
    off: np.ndarray            # int64 [P + 1]
    words: np.ndarray          # int32

    def wave(self, pi: int) -> np.ndarray:
        return self.words[self.off[pi]:self.off[pi + 1]]


def generate_testbench(spec: StimulusSpec) -> Testbench:
    """The edges generate_stimulus draws for the same spec, as one waveform per input
    over the whole testbench (absolute times cycle * period + offset)."""
    P, C, T, W = spec.num_inputs, spec.cycles, spec.period, spec.windows
    init, e_pi, e_cyc, e_off, _, _ = _draw_edges(spec)
    if C * T >= 2**31 - 1:
        raise ValueError("testbench longer than the int32 time range")
    cnt = np.bincount(e_pi, minlength=P)
    length = 1 + init + cnt + 1
    off = np.zeros(P + 1, dtype=np.int64)
    off[1:] = np.cumsum(length)
    words = np.empty(int(off[-1]), dtype=np.int32)
    s1 = off[:-1][init == 1]
    words[s1] = -1
    words[s1 + 1] = 0
    words[off[:-1][init == 0]] = 0
    first = np.zeros(P + 1, dtype=np.int64)
    first[1:] = np.cumsum(cnt)
    rank = np.arange(e_pi.size) - first[e_pi]
    words[(off[:-1] + 1 + init)[e_pi] + rank] = (e_cyc * T + e_off).astype(np.int32)
    words[off[1:] - 1] = EOW
    wc = window_cycles(C, W)
    return Testbench(num_inputs=P, num_windows=W, window_len=wc * T, window_cycles=wc, off=off, words=words)
