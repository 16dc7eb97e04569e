"""The C ABI library on the CPU: it loads, exports every entry point that
include/gatspi.h declares, and its host-side validation rejects bad netlists
before touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gatspi.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gatspi_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from gate_level_logic_gb300 import build
    build.build()
    from gate_level_logic_gb300 import gatspi
    return gatspi


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) == set(lib.SIGNATURES), "binding and header disagree"
    for n in names:
        assert callable(getattr(lib, n, None)), "no Python wrapper for " + n


def _struct(lib, net, W=1):
    keep = dict(lo=np.ascontiguousarray(net.level_offsets, np.int32), gt=np.ascontiguousarray(net.gate_type, np.int32),
                tp=np.ascontiguousarray(net.type_num_pins, np.int32), to=np.ascontiguousarray(net.type_tt_off, np.int32),
                tt=np.ascontiguousarray(net.tt_data, np.uint8), fo=np.ascontiguousarray(net.fanin_off, np.int32),
                fn=np.ascontiguousarray(net.fanin_net, np.int32), pw=np.ascontiguousarray(net.pin_weight, np.int32),
                wr=np.ascontiguousarray(net.wire_rise, np.int32), wf=np.ascontiguousarray(net.wire_fall, np.int32),
                do=np.ascontiguousarray(net.gate_dly_off, np.int64), dd=np.ascontiguousarray(net.dly_data, np.int32),
                wl=np.full(W, 100, np.int64))
    nl = lib.gatspi_netlist(net.num_inputs, net.num_gates, net.num_levels, len(keep["tp"]), keep["lo"].ctypes.data,
                            keep["gt"].ctypes.data, keep["tp"].ctypes.data, keep["to"].ctypes.data, keep["tt"].size,
                            keep["tt"].ctypes.data, keep["fo"].ctypes.data, keep["fn"].ctypes.data,
                            keep["pw"].ctypes.data, keep["wr"].ctypes.data, keep["wf"].ctypes.data,
                            keep["do"].ctypes.data, keep["dd"].size, keep["dd"].ctypes.data)
    cfg = lib.gatspi_config(W, keep["wl"].ctypes.data, 0, 0)
    return nl, cfg, keep


def _create_status(lib, nl, cfg, pool=0x10000, words=1024):
    ctx = ctypes.c_void_p()
    rc = lib.library().gatspi_create(ctypes.byref(nl), ctypes.byref(cfg), ctypes.c_void_p(pool), words,
                                     ctypes.byref(ctx))
    if rc == 0:
        lib.gatspi_destroy(ctx.value)
    return rc, lib.gatspi_last_error()


def _mutated(**changes):
    net, _ = synth.make("tiny")
    for k, v in changes.items():
        arr = getattr(net, k).copy()
        idx, val = v
        arr[idx] = val
        setattr(net, k, arr)
    return net


@pytest.mark.parametrize("change,needle", [
    (dict(fanin_net=(60 * 2, 150)), "not an input or a gate of a lower level"),   # gate 60 reads a later net
    (dict(pin_weight=(0, 3)), "pin weights"),
    (dict(wire_rise=(5, -1)), "interconnect delay"),
    (dict(wire_fall=(5, 70000)), "interconnect delay"),
    (dict(gate_type=(7, 99)), "type"),
    (dict(dly_data=(3, -5)), "delay"),
    (dict(level_offsets=(2, 250)), "level"),
])
def test_invalid_netlists_are_rejected_on_the_host(lib, change, needle):
    net = _mutated(**change)
    nl, cfg, keep = _struct(lib, net)
    rc, msg = _create_status(lib, nl, cfg)
    assert rc == 1 and needle in msg, (rc, msg)


def test_invalid_config_and_pool_are_rejected(lib):
    net, _ = synth.make("tiny")
    nl, cfg, keep = _struct(lib, net, W=1)
    assert _create_status(lib, nl, cfg, pool=0x10004)[0] == 1       # not 16-byte aligned
    assert _create_status(lib, nl, cfg, words=1023)[0] == 1         # not a multiple of 4 words
    cfg.num_windows = 0
    assert _create_status(lib, nl, cfg)[0] == 1
    # PATHPULSEPERCENT outside 0 .. 100, when the flag selects it
    for q in (-1, 101):
        nl, cfg, keep = _struct(lib, net, W=1)
        cfg.flags = lib.GATSPI_FLAG_PULSE_PERCENT
        cfg.pulse_percent = q
        rc, msg = _create_status(lib, nl, cfg)
        assert rc == 1 and "pulse_percent" in msg, (rc, msg)


def test_status_names(lib):
    for code, name in lib.STATUS.items():
        assert lib.gatspi_status_name(code) == name


def test_window_cutting_flags_on_the_host(lib):
    """The two window-cutting flags exclude each other (rejected before any device
    call), the binding's flag values are the header's, and the lanes query answers 0
    for no context."""
    net, _ = synth.make("tiny")
    nl, cfg, keep = _struct(lib, net, W=1)
    cfg.flags = lib.GATSPI_FLAG_WHOLE_WINDOWS | lib.GATSPI_FLAG_CUT_WINDOWS
    rc, msg = _create_status(lib, nl, cfg)
    assert rc == 1 and "exclude" in msg, (rc, msg)
    text = open(os.path.join(ROOT, "include", "gatspi.h")).read()
    for name, value in re.findall(r"#define (GATSPI_FLAG_[A-Z_]+) (0x[0-9a-f]+)u", text):
        assert getattr(lib, name) == int(value, 16), name
    for name in ("GATSPI_EOW", "GATSPI_NO_ARC", "GATSPI_MAX_PINS"):
        value = re.search(r"#define %s (\d+)" % name, text).group(1)
        assert getattr(lib, name) == int(value), name
    where = re.search(r"enum \{ GATSPI_HOST = (\d+), GATSPI_DEVICE = (\d+) \}", text)
    assert (lib.GATSPI_HOST, lib.GATSPI_DEVICE) == (int(where.group(1)), int(where.group(2)))
    assert lib.gatspi_lanes_per_window(0) == 0


def test_every_entry_point_cites_its_passage():
    """Each function of the C ABI is documented by the comment block above it (a struct
    of its arguments may stand in between), and that comment names the passage of the
    GATSPI page it implements or says that the page has no counterpart."""
    text = open(os.path.join(ROOT, "include", "gatspi.h")).read()
    passage = re.compile(r"Sections? \d|Fig\. \d|Algorithm 1|the page|no counterpart")
    names = declared_functions()
    assert len(names) >= 20
    for name in names:
        m = re.search(r"\n[a-z_0-9 ]+[ *]" + name + r"\s*\(", text)
        assert m, name
        before = text[:m.start()]
        start = before.rfind("/*")
        assert start >= 0 and before.rfind("*/") > start, name
        gap = before[before.rfind("*/") + 2:]
        assert gap.strip() == "" or gap.lstrip().startswith("typedef struct"), (name, gap[:80])
        comment = re.sub(r"\s*\n\s*\*?\s*", " ", before[start:])   # one line, margins dropped
        assert passage.search(comment), name


def test_product_path_does_not_use_the_oracle(lib):
    """The library and its binding neither import nor include anything under oracle/,
    and using them loads no oracle module: only the tests, smoke() and bench.py's
    CPU-baseline and reference legs run the oracle."""
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "gate_level_logic_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h", ".c")):
                with open(os.path.join(dirpath, f)) as fh:
                    text = fh.read()
                assert not re.search(r"^\s*(import oracle|from oracle)\b|#include\s*[\"<][^\">]*oracle", text, re.M), f
    code = ("import sys, numpy as np, synth\n"
            "from gate_level_logic_gb300 import gatspi, sdf_annotate\n"
            "net = synth.generate_netlist(synth.NetlistSpec(num_gates=200, num_inputs=8, num_levels=4, seed=1,\n"
            "                                              cond_cells=('AOI21',), cond_fraction=0.5))\n"
            "s = synth.write_sdf(net, seed=1)\n"
            "sdf_annotate(s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names, net.fanin_off,\n"
            "             net.gate_dly_off, net.dly_data.size, 1000)\n"
            "gatspi.gatspi_status_name(0)\n"
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]\n"
            "assert not bad, bad\n")
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT)


def test_missing_library_fails_loudly(lib, monkeypatch, tmp_path):
    """Without libgatspi.so every call of the binding raises: there is no CPU fallback
    to run instead."""
    monkeypatch.setattr(lib, "LIB_PATH", str(tmp_path / "libgatspi.so"))
    monkeypatch.setattr(lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        lib.library()
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        lib.gatspi_status_name(0)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        lib.gatspi_lanes_per_window(None)
