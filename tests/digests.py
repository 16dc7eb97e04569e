"""Digests for comparing runs too large to compare word by word (test infrastructure).

A net's digest is the 64-bit FNV-1a hash (one byte at a time) of the little-endian
bytes of its waveforms concatenated in window order, each window's Fig. 3 array
with its head and its EOW.  Two runs whose digests agree for every net have, up to
a 64-bit hash collision, the same words in every (net, window) waveform.

Per logic level the stored record holds exact sums (words, TC, T1) and three
position-keyed mixes: every gate's value is combined with its index by the
splitmix64 finaliser and the results are summed modulo 2^64, so a change of any
one gate's digest, TC or T1 (or two gates trading values) changes the mix.  The
same functions serve the oracle's digests (written by ``tests/golden/make_digests.py``)
and the CUDA library's (``gatspi_net_digests``) in the GPU tests.
"""
from __future__ import annotations

import functools
import hashlib

import numpy as np

import synth

FNV_OFFSET = np.uint64(14695981039346656037)
FNV_PRIME = np.uint64(1099511628211)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def fnv1a64(data: bytes, h: int = int(FNV_OFFSET)) -> int:
    """Plain 64-bit FNV-1a over bytes (pure Python)."""
    for b in data:
        h ^= b
        h = (h * int(FNV_PRIME)) & 0xFFFFFFFFFFFFFFFF
    return h


def net_digests(off, words, num_nets: int, num_windows: int) -> np.ndarray:
    """uint64 [num_nets]: the digest of every net from a CSR over (net, window)
    waveforms, net-major (the layout of the oracle's ``Result`` and of the library's
    gathered exports).  Vectorised across nets, byte by byte along each net."""
    off = np.asarray(off, np.int64)
    words = np.ascontiguousarray(words, np.int32)
    first = off[0:num_nets * num_windows:num_windows]
    last = off[num_windows:num_nets * num_windows + 1:num_windows]
    n = last - first
    h = np.full(num_nets, FNV_OFFSET, np.uint64)
    u = words.view(np.uint32)
    longest = int(n.max()) if num_nets else 0
    with np.errstate(over="ignore"):
        for k in range(longest):
            act = np.nonzero(n > k)[0]
            v = u[first[act] + k].astype(np.uint64)
            x = h[act]
            for b in range(4):
                x = (x ^ ((v >> np.uint64(8 * b)) & np.uint64(0xFF))) * FNV_PRIME
            h[act] = x
    return h


def mix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser, element-wise on uint64 (wrapping arithmetic)."""
    z = np.asarray(x, np.uint64).copy()
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def keyed_mix(values: np.ndarray, first_index: int = 0) -> int:
    """Sum over i of mix64(value_i + (first_index + i) * golden) modulo 2^64."""
    v = np.asarray(values).astype(np.int64).view(np.uint64)
    idx = np.arange(first_index, first_index + v.size, dtype=np.uint64)
    with np.errstate(over="ignore"):
        m = mix64(v + idx * _GOLDEN)
        return int(m.sum(dtype=np.uint64))


def level_records(level_offsets, num_inputs: int, net_hash, net_words, tc, t1) -> list:
    """One record per logic level (JSON-ready: 64-bit mixes as hex strings)."""
    lo = np.asarray(level_offsets, np.int64)
    out = []
    for lvl in range(lo.size - 1):
        g0, g1 = int(lo[lvl]), int(lo[lvl + 1])
        n0, n1 = num_inputs + g0, num_inputs + g1
        out.append({
            "gates": g1 - g0,
            "words": int(np.asarray(net_words[n0:n1], np.int64).sum()),
            "tc": int(np.asarray(tc[g0:g1], np.int64).sum()),
            "t1": int(np.asarray(t1[g0:g1], np.int64).sum()),
            "tc_mix": "%016x" % keyed_mix(tc[g0:g1], g0),
            "t1_mix": "%016x" % keyed_mix(t1[g0:g1], g0),
            "wave_mix": "%016x" % keyed_mix(np.asarray(net_hash[n0:n1], np.uint64).view(np.int64), n0),
        })
    return out


def input_record(num_inputs: int, net_hash, net_words) -> dict:
    return {
        "words": int(np.asarray(net_words[:num_inputs], np.int64).sum()),
        "wave_mix": "%016x" % keyed_mix(np.asarray(net_hash[:num_inputs], np.uint64).view(np.int64), 0),
    }


def inputs_sha256(net, stim) -> str:
    """Digest of the generated netlist and stimulus arrays (detects a generator that
    drew different inputs on another machine)."""
    h = hashlib.sha256()
    for a in (net.level_offsets, net.gate_type, net.type_num_pins, net.type_tt_off, net.tt_data, net.fanin_off,
              net.fanin_net, net.pin_weight, net.wire_rise, net.wire_fall, net.gate_dly_off, net.dly_data,
              stim.window_len, stim.pi_off, stim.pi_words):
        a = np.ascontiguousarray(a)
        h.update(str(a.dtype).encode())
        h.update(np.asarray(a.shape, np.int64).tobytes())
        h.update(a.tobytes())
    return h.hexdigest()


@functools.lru_cache(maxsize=1)
def _sweep_netlist():
    net_kw, _ = synth.WORKLOADS["1M"]
    return synth.generate_netlist(synth.NetlistSpec(**net_kw))


def _sweep_point(activity, windows):
    """synth.sweep(activity, windows) with the 1M-gate netlist generated once."""
    _, stim_kw = synth.WORKLOADS["1M"]
    kw = dict(stim_kw, activity=activity, windows=windows, seed=4, glitch_frac=0.0)
    return _sweep_netlist(), synth.generate_stimulus(synth.StimulusSpec(**kw))


def large_workloads() -> dict:
    """The full-size workloads with stored oracle digests: name -> (description,
    maker of (net, stim))."""
    out = {
        "5M": ("5M gates, 60 levels, 30% conditional arcs; 16384 inputs, 2000 cycles, 20%, 128 windows",
               lambda: synth.make("5M")),
        "scan500k": ("500k NAND2/NOR2/XOR2 gates, 30 levels; 4096 inputs, 100k cycles, 2%, 256 windows",
                     lambda: synth.make("scan500k")),
    }
    for a in synth.SWEEP_ACTIVITY:
        for w in synth.SWEEP_WINDOWS:
            out["sweep-%g-%d" % (a, w)] = (
                "1M-gate netlist, stimulus seed 4, %g%% activity, no glitch pairs, %d windows" % (100 * a, w),
                (lambda a=a, w=w: _sweep_point(a, w)))
    # below PATHPULSEPERCENT 100, where few long windows are cut into time chunks: one
    # window (at 50 % its heavy gates are split into segments) and sixteen at 0
    # (transport delay)
    for a, w, q in ((0.05, 1, 50), (0.5, 1, 50), (0.2, 16, 0)):
        out["sweep-%g-%d-q%d" % (a, w, q)] = (
            "1M-gate netlist, stimulus seed 4, %g%% activity, no glitch pairs, %d windows, PATHPULSEPERCENT %d"
            % (100 * a, w, q), (lambda a=a, w=w: _sweep_point(a, w)))
    return out


def pulse_percent(name: str) -> int:
    """PATHPULSEPERCENT of a stored workload: its name's '-qN' suffix, else 100."""
    return int(name.rsplit("-q", 1)[1]) if "-q" in name else 100
