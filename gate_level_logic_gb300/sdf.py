"""SDF text -> delay tables and interconnect delays, through the library's native
translator (gatspi_sdf_annotate; GATSPI page, Section 3, Fig. 4)."""
from __future__ import annotations

import ctypes

import numpy as np

from . import gatspi as _c


def _strings(items):
    enc = [s.encode() for s in items]
    arr = (ctypes.c_char_p * max(len(enc), 1))(*enc)
    return arr, enc


def sdf_annotate(text, type_names, type_pins, gate_type, instance_names, fanin_off, gate_dly_off, dly_len,
                 unit_fs=1000, out_pin="Y"):
    """(dly_data int32 [dly_len], wire_rise int32 [E], wire_fall int32 [E]) from SDF text.

    type_pins[t]: type t's input pin names in pin order; instance_names[g]: gate g's
    SDF instance; fanin_off[G+1]: each gate's fanin edges; gate_dly_off[G]: where its
    [4n][2^(n-1)] table goes; unit_fs: the simulator's time unit in femtoseconds."""
    gate_type = np.ascontiguousarray(gate_type, np.int32)
    fanin_off = np.ascontiguousarray(fanin_off, np.int32)
    gate_dly_off = np.ascontiguousarray(gate_dly_off, np.int64)
    num_pins = np.ascontiguousarray([len(p) for p in type_pins], np.int32)
    tn, tn_keep = _strings(type_names)
    pn, pn_keep = _strings([p for pins in type_pins for p in pins])
    inst, inst_keep = _strings(instance_names)
    G = int(gate_type.size)
    design = _c.gatspi_sdf_design(len(type_names), ctypes.addressof(tn), num_pins.ctypes.data, ctypes.addressof(pn),
                                  out_pin.encode(), G, gate_type.ctypes.data, ctypes.addressof(inst),
                                  fanin_off.ctypes.data, gate_dly_off.ctypes.data, int(dly_len), int(unit_fs))
    E = int(fanin_off[G]) if G else 0
    dly = np.zeros(max(int(dly_len), 1), np.int32)
    wr = np.zeros(max(E, 1), np.int32)
    wf = np.zeros(max(E, 1), np.int32)
    data = text.encode() if isinstance(text, str) else bytes(text)
    _c.gatspi_sdf_annotate(design, data, dly.ctypes.data, wr.ctypes.data, wf.ctypes.data)
    return dly[:int(dly_len)], wr[:E], wf[:E]
