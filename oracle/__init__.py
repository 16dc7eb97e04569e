"""CPU oracle of the gate-level re-simulator -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
binding) never does; the two share no code.

Two independent CPU simulators, both plain C compiled with gcc:

* ``simulate`` -- the serial event-driven simulator that follows Algorithm 1 of
  the GATSPI page (Section 3) gate by gate in level order and window by window
  (optionally with windows spread over threads; windows are independent);
* ``bruteforce`` -- a unit-time-step simulator of inertial wire and gate
  elements, used to pin ``simulate`` on tiny netlists;
* ``digest`` -- the same Algorithm 1 run (a level-parallel driver around the same
  per-task routine) that keeps no merged pool and returns a 64-bit FNV-1a digest of
  every net's waveforms instead, continued over consecutive batches of windows, for
  runs too large to compare word by word.

And the testbench restructuring: ``restructure`` cuts whole-testbench input
waveforms into the cycle windows (GATSPI page, Sections 1, 4 and 5).

Both return the same layout: CSR offsets over every (net, window) waveform,
net-major and window-minor, into a pool that holds the input waveforms followed by
the gate outputs; plus per-gate toggle counts TC and time-at-1 T1 summed over
windows (T0 = total window time - T1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SOURCES = ("gatspi_oracle.c", "bruteforce.c", "testbench.c")
_libs = {}


def build(force: bool = False, src_dir: str = _HERE, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc into ``out`` (default ``oracle/liboracle.so``)."""
    srcs = [os.path.join(src_dir, s) for s in _SOURCES]
    hdr = os.path.join(src_dir, "oracle_abi.h")
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(p) for p in srcs + [hdr])
        if os.path.getmtime(out) >= newest:
            return out
    tmp = out + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-Wall", "-Wextra", "-pthread",
           "-shared", "-fPIC", "-o", tmp] + srcs
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


class _Net(ctypes.Structure):
    _fields_ = [
        ("num_inputs", ctypes.c_int32), ("num_gates", ctypes.c_int32),
        ("num_levels", ctypes.c_int32), ("num_types", ctypes.c_int32),
        ("level_offsets", ctypes.c_void_p), ("gate_type", ctypes.c_void_p),
        ("type_num_pins", ctypes.c_void_p), ("type_tt_off", ctypes.c_void_p),
        ("tt_data", ctypes.c_void_p), ("fanin_off", ctypes.c_void_p),
        ("fanin_net", ctypes.c_void_p), ("pin_weight", ctypes.c_void_p),
        ("wire_rise", ctypes.c_void_p), ("wire_fall", ctypes.c_void_p),
        ("gate_dly_off", ctypes.c_void_p), ("dly_data", ctypes.c_void_p),
    ]


def _load(path=None):
    path = path or _LIB_PATH
    if path not in _libs:
        if path == _LIB_PATH:
            build()
        lib = ctypes.CDLL(path)
        sig = [ctypes.POINTER(_Net), ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
               ctypes.c_int32]
        lib.oracle_simulate.argtypes = sig + [ctypes.c_int, ctypes.c_void_p,
                                              ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int64),
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int]
        lib.oracle_simulate.restype = ctypes.c_int
        lib.brute_simulate.argtypes = sig + [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
                                             ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_char_p, ctypes.c_int]
        lib.brute_simulate.restype = ctypes.c_int
        lib.oracle_restructure.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
                                           ctypes.POINTER(ctypes.c_int64), ctypes.c_char_p, ctypes.c_int]
        lib.oracle_restructure.restype = ctypes.c_int
        lib.oracle_digest.argtypes = sig + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int]
        lib.oracle_digest.restype = ctypes.c_int
        lib.oracle_fnv1a64.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_fnv1a64.restype = ctypes.c_uint64
        lib.oracle_free.argtypes = [ctypes.c_void_p]
        lib.oracle_set_literal_skip.argtypes = [ctypes.c_int]
        lib.oracle_set_literal_skip.restype = None
        lib.oracle_free.restype = None
        _libs[path] = lib
    return _libs[path]


class OracleError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("oracle error %d: %s" % (code, msg))
        self.code = code


@dataclass
class Result:
    off: np.ndarray    # int64 [(P+G)*W + 1]
    pool: np.ndarray   # int32
    tc: np.ndarray     # int64 [G]
    t1: np.ndarray     # int64 [G]
    t0: np.ndarray     # int64 [G]
    num_inputs: int
    num_windows: int

    def wave(self, net: int, w: int) -> np.ndarray:
        k = net * self.num_windows + w
        return self.pool[self.off[k]:self.off[k + 1]]

    def gate_wave(self, g: int, w: int) -> np.ndarray:
        return self.wave(self.num_inputs + g, w)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _marshal(net, stim):
    keep = dict(
        level_offsets=_c(net.level_offsets, np.int32), gate_type=_c(net.gate_type, np.int32),
        type_num_pins=_c(net.type_num_pins, np.int32), type_tt_off=_c(net.type_tt_off, np.int32),
        tt_data=_c(net.tt_data, np.uint8), fanin_off=_c(net.fanin_off, np.int32),
        fanin_net=_c(net.fanin_net, np.int32), pin_weight=_c(net.pin_weight, np.int32),
        wire_rise=_c(net.wire_rise, np.int32), wire_fall=_c(net.wire_fall, np.int32),
        gate_dly_off=_c(net.gate_dly_off, np.int64), dly_data=_c(net.dly_data, np.int32),
        window_len=_c(stim.window_len, np.int64), pi_off=_c(stim.pi_off, np.int64),
        pi_words=_c(stim.pi_words, np.int32),
    )
    s = _Net(net.num_inputs, net.num_gates, net.num_levels, len(net.type_num_pins),
             *[keep[k].ctypes.data for k in ("level_offsets", "gate_type", "type_num_pins", "type_tt_off",
                                              "tt_data", "fanin_off", "fanin_net", "pin_weight", "wire_rise",
                                              "wire_fall", "gate_dly_off", "dly_data")])
    return s, keep


def _finish(lib, rc, err, pool_ptr, pool_words, off, tc, t1, net, stim):
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    n = int(pool_words.value)
    try:
        buf = (ctypes.c_int32 * max(n, 1)).from_address(pool_ptr.value)
        pool = np.frombuffer(buf, dtype=np.int32, count=n).copy()
    finally:
        lib.oracle_free(pool_ptr)
    t0 = int(np.asarray(stim.window_len, dtype=np.int64).sum()) - t1
    return Result(off=off, pool=pool, tc=tc, t1=t1, t0=t0, num_inputs=net.num_inputs,
                  num_windows=stim.num_windows)


def simulate(net, stim, threads: int = 1, lib_path: str = None, pulse_percent: int = 100,
             literal_skip: bool = False) -> Result:
    """Event-driven oracle (Algorithm 1) over all gates and windows.  ``pulse_percent``
    is PATHPULSEPERCENT: the inertial reject limit of both filters as a percentage of
    the delay (100 = the page's setting, 0 = transport delay).  ``literal_skip`` runs
    the study variant of the interconnect pulse test: one test per pin and iteration
    of the event loop, as Algorithm 1 writes it, instead of skipping every narrow pulse
    in a row (the reading the rest of the project computes)."""
    lib = _load(lib_path)
    if literal_skip:
        lib.oracle_set_literal_skip(1)
        try:
            return simulate(net, stim, threads, lib_path, pulse_percent)
        finally:
            lib.oracle_set_literal_skip(0)
    s, keep = _marshal(net, stim)
    W = int(stim.num_windows)
    off = np.zeros((net.num_inputs + net.num_gates) * W + 1, dtype=np.int64)
    tc = np.zeros(max(net.num_gates, 1), dtype=np.int64)
    t1 = np.zeros(max(net.num_gates, 1), dtype=np.int64)
    pool_ptr, pool_words = ctypes.c_void_p(), ctypes.c_int64()
    err = ctypes.create_string_buffer(512)
    rc = lib.oracle_simulate(ctypes.byref(s), W, keep["window_len"].ctypes.data, keep["pi_off"].ctypes.data,
                             keep["pi_words"].ctypes.data, int(pulse_percent), int(threads), off.ctypes.data,
                             ctypes.byref(pool_ptr), ctypes.byref(pool_words), tc.ctypes.data, t1.ctypes.data,
                             err, 512)
    return _finish(lib, rc, err, pool_ptr, pool_words, off, tc[:net.num_gates], t1[:net.num_gates], net, stim)


def bruteforce(net, stim, lib_path: str = None, pulse_percent: int = 100) -> Result:
    """Unit-time-step inertial-element simulator (tiny cases only)."""
    lib = _load(lib_path)
    s, keep = _marshal(net, stim)
    W = int(stim.num_windows)
    off = np.zeros((net.num_inputs + net.num_gates) * W + 1, dtype=np.int64)
    tc = np.zeros(max(net.num_gates, 1), dtype=np.int64)
    t1 = np.zeros(max(net.num_gates, 1), dtype=np.int64)
    pool_ptr, pool_words = ctypes.c_void_p(), ctypes.c_int64()
    err = ctypes.create_string_buffer(512)
    rc = lib.brute_simulate(ctypes.byref(s), W, keep["window_len"].ctypes.data, keep["pi_off"].ctypes.data,
                            keep["pi_words"].ctypes.data, int(pulse_percent), off.ctypes.data, ctypes.byref(pool_ptr),
                            ctypes.byref(pool_words), tc.ctypes.data, t1.ctypes.data, err, 512)
    return _finish(lib, rc, err, pool_ptr, pool_words, off, tc[:net.num_gates], t1[:net.num_gates], net, stim)


def restructure(tb_off, tb_words, window_len, lib_path: str = None):
    """Cut whole-testbench input waveforms (CSR ``tb_off[P+1]`` over ``tb_words``) into
    windows of ``window_len`` time units.  Returns ``(off, words)``: CSR offsets over the
    (input, window) waveforms, input-major and window-minor, and their words."""
    lib = _load(lib_path)
    tb_off = _c(tb_off, np.int64)
    tb_words = _c(tb_words, np.int32)
    wl = _c(window_len, np.int64).reshape(-1)
    P, W = tb_off.size - 1, wl.size
    off = np.zeros(P * W + 1, dtype=np.int64)
    ptr, n = ctypes.c_void_p(), ctypes.c_int64()
    err = ctypes.create_string_buffer(512)
    rc = lib.oracle_restructure(P, tb_off.ctypes.data, tb_words.ctypes.data, W, wl.ctypes.data, off.ctypes.data,
                                ctypes.byref(ptr), ctypes.byref(n), err, 512)
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    try:
        buf = (ctypes.c_int32 * max(int(n.value), 1)).from_address(ptr.value)
        words = np.frombuffer(buf, dtype=np.int32, count=int(n.value)).copy()
    finally:
        lib.oracle_free(ptr)
    return off, words


FNV_OFFSET = 14695981039346656037


@dataclass
class Digest:
    """Running digests of a run done in consecutive batches of windows."""
    net_hash: np.ndarray    # uint64 [P+G]: FNV-1a of each net's waveforms so far, window order
    net_words: np.ndarray   # int64 [P+G]: words hashed so far
    tc: np.ndarray          # int64 [G]
    t1: np.ndarray          # int64 [G]
    window_time: int        # sum of the window lengths so far (T0 = window_time - T1)

    @classmethod
    def start(cls, num_inputs: int, num_gates: int) -> "Digest":
        n = num_inputs + num_gates
        return cls(net_hash=np.full(n, FNV_OFFSET, np.uint64), net_words=np.zeros(n, np.int64),
                   tc=np.zeros(num_gates, np.int64), t1=np.zeros(num_gates, np.int64), window_time=0)


def digest(net, stim, state: Digest = None, threads: int = 1, lib_path: str = None,
           pulse_percent: int = 100) -> Digest:
    """Algorithm 1 over every gate and window of ``stim`` (levels in order, a level's
    (gate, window) tasks spread over ``threads``); continues ``state`` (a new one if
    None) with this batch of windows, which must follow the windows already in it."""
    lib = _load(lib_path)
    s, keep = _marshal(net, stim)
    if state is None:
        state = Digest.start(net.num_inputs, net.num_gates)
    G = net.num_gates
    tc = np.zeros(max(G, 1), np.int64)
    t1 = np.zeros(max(G, 1), np.int64)
    h = np.ascontiguousarray(state.net_hash, np.uint64).copy()
    nw = np.ascontiguousarray(state.net_words, np.int64).copy()
    err = ctypes.create_string_buffer(512)
    rc = lib.oracle_digest(ctypes.byref(s), int(stim.num_windows), keep["window_len"].ctypes.data,
                           keep["pi_off"].ctypes.data, keep["pi_words"].ctypes.data, int(pulse_percent), int(threads),
                           h.ctypes.data, nw.ctypes.data, tc.ctypes.data, t1.ctypes.data, err, 512)
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return Digest(net_hash=h, net_words=nw, tc=state.tc + tc[:G], t1=state.t1 + t1[:G],
                  window_time=state.window_time + int(np.asarray(stim.window_len, np.int64).sum()))


def fnv1a64(data: bytes, h: int = FNV_OFFSET, lib_path: str = None) -> int:
    """The oracle's 64-bit FNV-1a over raw bytes (for pinning it on published vectors)."""
    lib = _load(lib_path)
    buf = ctypes.create_string_buffer(bytes(data), max(len(data), 1))
    return int(lib.oracle_fnv1a64(ctypes.c_uint64(h), buf, len(data)))
