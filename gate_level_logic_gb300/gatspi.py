"""ctypes binding of the C ABI in include/gatspi.h (argument marshalling only).

Every function keeps the C name.  Nothing here simulates: every step of the
re-simulation runs in the CUDA library ``libgatspi.so``; if that library is missing
the import fails loudly (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgatspi.so")

GATSPI_EOW = 2147483647
GATSPI_NO_ARC = 2147483647
GATSPI_MAX_PINS = 4
GATSPI_HOST, GATSPI_DEVICE = 0, 1
GATSPI_FLAG_LEVEL_TIMING = 0x1
GATSPI_FLAG_NO_GRAPH = 0x2
GATSPI_FLAG_PULSE_PERCENT = 0x4
GATSPI_FLAG_COMPACT = 0x8
GATSPI_FLAG_WHOLE_WINDOWS = 0x10
GATSPI_FLAG_CUT_WINDOWS = 0x20

STATUS = {
    0: "GATSPI_OK", 1: "GATSPI_EINVAL", 2: "GATSPI_ENOMEM", 3: "GATSPI_EPOOL_OVERFLOW", 4: "GATSPI_EBADWAVE",
    5: "GATSPI_ECUDA", 6: "GATSPI_ESTATE", 7: "GATSPI_EBADLUT", 8: "GATSPI_ETIMEOUT", 9: "GATSPI_EINTERNAL",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

_p = ctypes.c_void_p


class gatspi_netlist(ctypes.Structure):
    _fields_ = [
        ("num_inputs", ctypes.c_int32), ("num_gates", ctypes.c_int32), ("num_levels", ctypes.c_int32),
        ("num_types", ctypes.c_int32), ("level_offsets", _p), ("gate_type", _p), ("type_num_pins", _p),
        ("type_tt_off", _p), ("tt_len", ctypes.c_int64), ("tt_data", _p), ("fanin_off", _p), ("fanin_net", _p),
        ("pin_weight", _p), ("wire_rise", _p), ("wire_fall", _p), ("gate_dly_off", _p), ("dly_len", ctypes.c_int64),
        ("dly_data", _p),
    ]


class gatspi_config(ctypes.Structure):
    _fields_ = [("num_windows", ctypes.c_int32), ("window_len", _p), ("flags", ctypes.c_uint32),
                ("pulse_percent", ctypes.c_int32)]


class gatspi_views(ctypes.Structure):
    _fields_ = [
        ("pool", _p), ("pool_words", ctypes.c_int64), ("pool_used", ctypes.c_int64), ("net_base", _p),
        ("wstart", _p), ("wend", _p), ("tc", _p), ("t1", _p), ("num_nets", ctypes.c_int32),
        ("num_windows", ctypes.c_int32),
    ]


class gatspi_level_args(ctypes.Structure):
    _fields_ = [
        ("gate_desc", _p), ("dly_data", _p), ("window_len", _p), ("pool", _p),
        ("pool_words", ctypes.c_int64), ("net_base", _p), ("wstart", _p), ("wend", _p), ("wlen8", _p), ("perm", _p),
        ("goff", _p),
        ("tc", _p), ("t1", _p),
        ("level_base", _p), ("num_inputs", ctypes.c_int32), ("num_windows", ctypes.c_int32),
        ("gate_begin", ctypes.c_int32), ("num_gates", ctypes.c_int32),
        ("flags", ctypes.c_uint32), ("pulse_percent", ctypes.c_int32),
    ]


class gatspi_sdf_design(ctypes.Structure):
    _fields_ = [
        ("num_types", ctypes.c_int32), ("type_names", _p), ("type_num_pins", _p), ("pin_names", _p),
        ("out_pin", ctypes.c_char_p), ("num_gates", ctypes.c_int32), ("gate_type", _p), ("instance_names", _p),
        ("fanin_off", _p), ("gate_dly_off", _p), ("dly_len", ctypes.c_int64), ("unit_fs", ctypes.c_int64),
    ]


# exported symbol -> (restype, argtypes)
SIGNATURES = {
    "gatspi_create": (ctypes.c_int, [ctypes.POINTER(gatspi_netlist), ctypes.POINTER(gatspi_config), _p, ctypes.c_size_t,
                                     ctypes.POINTER(_p)]),
    "gatspi_load_waveforms": (ctypes.c_int, [_p, _p, _p, ctypes.c_size_t, ctypes.c_int, _p]),
    "gatspi_load_testbench": (ctypes.c_int, [_p, _p, _p, ctypes.c_size_t, ctypes.c_int, _p]),
    "gatspi_simulate": (ctypes.c_int, [_p, _p]),
    "gatspi_sync": (ctypes.c_int, [_p]),
    "gatspi_lanes_per_window": (ctypes.c_int32, [_p]),
    "gatspi_toggle_stats": (ctypes.c_int, [_p, _p, _p, _p]),
    "gatspi_toggle_stats_host": (ctypes.c_int, [_p, ctypes.POINTER(_p), ctypes.POINTER(_p), ctypes.POINTER(ctypes.c_int64)]),
    "gatspi_input_stats": (ctypes.c_int, [_p, _p, _p, _p]),
    "gatspi_write_saif": (ctypes.c_int, [_p, ctypes.c_char_p, ctypes.c_char_p, ctypes.c_char_p, _p]),
    "gatspi_get_waveform": (ctypes.c_int, [_p, ctypes.c_int32, ctypes.c_int32, _p, ctypes.c_size_t,
                                           ctypes.POINTER(ctypes.c_size_t)]),
    "gatspi_export_offsets": (ctypes.c_int, [_p, _p, _p, ctypes.c_size_t]),
    "gatspi_export_windows": (ctypes.c_int, [_p, _p, ctypes.c_int32, _p, _p, ctypes.c_size_t]),
    "gatspi_net_digests": (ctypes.c_int, [_p, ctypes.c_int64, ctypes.c_int64, _p, _p]),
    "gatspi_device_views": (ctypes.c_int, [_p, ctypes.POINTER(gatspi_views)]),
    "gatspi_level_times": (ctypes.c_int, [_p, _p, _p, ctypes.c_int32]),
    "gatspi_set_level_timing": (ctypes.c_int, [_p, ctypes.c_int32]),
    "gatspi_simulate_level_static": (ctypes.c_int, [ctypes.POINTER(gatspi_level_args), _p]),
    "gatspi_sdf_annotate": (ctypes.c_int, [ctypes.POINTER(gatspi_sdf_design), ctypes.c_char_p, ctypes.c_size_t, _p,
                                           _p, _p]),
    "gatspi_inject_scan_stall": (ctypes.c_int, [_p, ctypes.c_int32, ctypes.c_int64]),
    "gatspi_destroy": (None, [_p]),
    "gatspi_last_error": (ctypes.c_char_p, []),
    "gatspi_status_name": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def library():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgatspi.so is missing: build it with gate_level_logic_gb300.build.build() "
                               "(needs nvcc); there is no CPU fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class GatspiError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status
        self.name = STATUS.get(status, str(status))


def _check(rc: int):
    if rc != 0:
        raise GatspiError(rc, library().gatspi_last_error().decode(errors="replace"))


def gatspi_create(nl: gatspi_netlist, cfg: gatspi_config, d_pool: int, pool_words: int) -> int:
    ctx = _p()
    _check(library().gatspi_create(ctypes.byref(nl), ctypes.byref(cfg), _p(d_pool), pool_words, ctypes.byref(ctx)))
    return ctx.value


def gatspi_load_waveforms(ctx: int, off: int, words: int, nwords: int, where: int, stream: int = 0):
    _check(library().gatspi_load_waveforms(_p(ctx), _p(off), _p(words), nwords, where, _p(stream)))


def gatspi_load_testbench(ctx: int, off: int, words: int, nwords: int, where: int, stream: int = 0):
    _check(library().gatspi_load_testbench(_p(ctx), _p(off), _p(words), nwords, where, _p(stream)))


def gatspi_simulate(ctx: int, stream: int = 0):
    _check(library().gatspi_simulate(_p(ctx), _p(stream)))


def gatspi_sync(ctx: int):
    _check(library().gatspi_sync(_p(ctx)))


def gatspi_lanes_per_window(ctx: int) -> int:
    """Lanes the next simulate gives each window: 32 // W when it cuts windows into
    time chunks, else 1."""
    return int(library().gatspi_lanes_per_window(_p(ctx)))


def gatspi_toggle_stats(ctx: int, tc: int, t0: int, t1: int):
    _check(library().gatspi_toggle_stats(_p(ctx), _p(tc), _p(t0), _p(t1)))


def gatspi_toggle_stats_host(ctx: int):
    """(tc pointer, t1 pointer, sum of window lengths)."""
    tc, t1, ws = _p(), _p(), ctypes.c_int64()
    _check(library().gatspi_toggle_stats_host(_p(ctx), ctypes.byref(tc), ctypes.byref(t1), ctypes.byref(ws)))
    return tc.value or 0, t1.value or 0, ws.value


def gatspi_input_stats(ctx: int, tc: int, t0: int, t1: int):
    _check(library().gatspi_input_stats(_p(ctx), _p(tc), _p(t0), _p(t1)))


def gatspi_write_saif(ctx: int, path: str, design: str = None, timescale: str = None, net_names: int = 0):
    enc = (lambda x: None if x is None else x.encode())
    _check(library().gatspi_write_saif(_p(ctx), enc(path), enc(design), enc(timescale), _p(net_names)))


def gatspi_get_waveform(ctx: int, net: int, window: int, buf: int, cap: int) -> int:
    n = ctypes.c_size_t()
    rc = library().gatspi_get_waveform(_p(ctx), net, window, _p(buf), cap, ctypes.byref(n))
    if rc != 0 and not (rc == 1 and n.value > cap):
        _check(rc)
    return n.value


def gatspi_export_offsets(ctx: int, start: int, length: int, n: int):
    _check(library().gatspi_export_offsets(_p(ctx), _p(start), _p(length), n))


def gatspi_export_windows(ctx: int, windows: int, nsel: int, off: int, words: int, cap: int):
    _check(library().gatspi_export_windows(_p(ctx), _p(windows), nsel, _p(off), _p(words), cap))


def gatspi_net_digests(ctx: int, net_begin: int, num_nets: int, digest: int, words: int = 0):
    _check(library().gatspi_net_digests(_p(ctx), net_begin, num_nets, _p(digest), _p(words)))


def gatspi_device_views(ctx: int) -> gatspi_views:
    v = gatspi_views()
    _check(library().gatspi_device_views(_p(ctx), ctypes.byref(v)))
    return v


def gatspi_level_times(ctx: int, sim_ms: int, bounds_ms: int, n: int):
    _check(library().gatspi_level_times(_p(ctx), _p(sim_ms), _p(bounds_ms), n))


def gatspi_set_level_timing(ctx: int, on: bool):
    _check(library().gatspi_set_level_timing(_p(ctx), 1 if on else 0))


def gatspi_simulate_level_static(args: gatspi_level_args, stream: int = 0):
    _check(library().gatspi_simulate_level_static(ctypes.byref(args), _p(stream)))


def gatspi_sdf_annotate(design: gatspi_sdf_design, text: bytes, dly_data: int, wire_rise: int = 0,
                        wire_fall: int = 0):
    _check(library().gatspi_sdf_annotate(ctypes.byref(design), text, len(text), _p(dly_data), _p(wire_rise),
                                         _p(wire_fall)))


def gatspi_inject_scan_stall(ctx: int, level: int, wait_ns: int):
    _check(library().gatspi_inject_scan_stall(_p(ctx), level, wait_ns))


def gatspi_destroy(ctx: int):
    library().gatspi_destroy(_p(ctx))


def gatspi_last_error() -> str:
    return library().gatspi_last_error().decode(errors="replace")


def gatspi_status_name(status: int) -> str:
    return library().gatspi_status_name(status).decode()
