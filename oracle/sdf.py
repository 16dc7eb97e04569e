"""TEST INFRASTRUCTURE ONLY: the oracle's SDF-to-delay-table translation.

Only tests/ and bench.py's CPU-baseline leg may import this module.  It shares no
code with the library's translator and is deliberately plain and slow.

What it computes (GATSPI: GPU-Accelerated Gate-Level Simulation for Power
Improvement, Section 3 and Fig. 4): SDF delay statements turned into the per-
instance 2-D delay arrays the simulator looks up.  A row is a switching pin with its
input edge and the output edge: row = 4 * pin + 2 * e_in + e_out with RISE = 0 and
FALL = 1; a column is the values of the other pins, in pin order with the first one
most significant (Fig. 4: for AOI21 B -> Y, A1 weighs 2 and A2 weighs 1).

Readings where the page is silent:
  - (IOPATH (posedge P) Y r f) sets the rows of pin P with e_in = RISE, (negedge P)
    those with e_in = FALL, a bare P both; r is the output-rise delay and f the
    output-fall delay (with one value it serves both); an empty () means no arc,
    written INT32_MAX;
  - an IOPATH without COND sets every column; (COND expr (IOPATH ...)) sets the
    columns where expr holds for the other pins' values, over the unconditional
    statement whatever the order; where several COND statements hold, the one
    written last wins;
  - a min:typ:max triple gives its typ value; values are in the file's TIMESCALE and
    are converted to the simulator's unit exactly, then rounded to the nearest
    integer (halves up); negative values are rejected;
  - (INTERCONNECT src inst/pin r f) sets that pin's wire rise and fall delays; pins
    without one keep 0;
  - rows that no statement sets stay INT32_MAX; a file without TIMESCALE is in 1 ns
    (SDF's default).
Conditions are Verilog expressions over the other pins: ``== === != !==``,
``! ~ & | ^ && ||``, parentheses, the literals 0, 1, 1'b0, 1'b1, 'b0, 'b1.
"""
from __future__ import annotations

import re
from fractions import Fraction

import numpy as np

INF = 2**31 - 1
_FS = {"s": 10**15, "ms": 10**12, "us": 10**9, "ns": 10**6, "ps": 10**3, "fs": 1}


class SdfError(ValueError):
    pass


# ---- S-expressions ---------------------------------------------------------------

def _tokens(text):
    return re.findall(r'\(|\)|"[^"]*"|[^\s()]+', text)


def _tree(text):
    toks = _tokens(text)
    stack = [[]]
    for t in toks:
        if t == "(":
            stack.append([])
        elif t == ")":
            if len(stack) == 1:
                raise SdfError("unbalanced parentheses")
            done = stack.pop()
            stack[-1].append(done)
        else:
            stack[-1].append(t)
    if len(stack) != 1 or len(stack[0]) != 1:
        raise SdfError("unbalanced parentheses")
    return stack[0][0]


def _flatten(items):
    """Expression items (atoms and nested lists) back to text."""
    out = []
    for it in items:
        out.append("(" + _flatten(it) + ")" if isinstance(it, list) else it)
    return " ".join(out)


# ---- conditions ------------------------------------------------------------------

_EXPR_TOKEN = re.compile(r"\s*(===|!==|==|!=|&&|\|\||[!~&|^()]|\d*'[bB][01]|[01]\b|[A-Za-z_][A-Za-z0-9_\[\]\\.]*)")


class _Cond:
    """Parsed condition; value(env) evaluates it for 0/1 pin values."""

    def __init__(self, text):
        pos, self.toks = 0, []
        text = text.strip()
        while pos < len(text):
            m = _EXPR_TOKEN.match(text, pos)
            if not m or m.end() == pos:
                raise SdfError("bad condition: %r" % text)
            self.toks.append(m.group(1))
            pos = m.end()
            while pos < len(text) and text[pos].isspace():
                pos += 1
        self.names = {t for t in self.toks if re.match(r"[A-Za-z_]", t)}

    def value(self, env):
        self.k = 0
        self.env = env
        v = self._or()
        if self.k != len(self.toks):
            raise SdfError("bad condition: %r" % " ".join(self.toks))
        return v

    def _peek(self):
        return self.toks[self.k] if self.k < len(self.toks) else None

    def _take(self):
        self.k += 1
        return self.toks[self.k - 1]

    def _binary(self, ops, sub):
        v = sub()
        while self._peek() in ops:
            op = self._take()
            w = sub()
            if op == "||":
                v = int(bool(v) or bool(w))
            elif op == "&&":
                v = int(bool(v) and bool(w))
            elif op == "|":
                v = v | w
            elif op == "^":
                v = v ^ w
            elif op == "&":
                v = v & w
            elif op in ("==", "==="):
                v = int(v == w)
            else:
                v = int(v != w)
        return v

    def _or(self):
        return self._binary(("||",), self._and)

    def _and(self):
        return self._binary(("&&",), self._bor)

    def _bor(self):
        return self._binary(("|",), self._bxor)

    def _bxor(self):
        return self._binary(("^",), self._band)

    def _band(self):
        return self._binary(("&",), self._eq)

    def _eq(self):
        return self._binary(("==", "===", "!=", "!=="), self._unary)

    def _unary(self):
        t = self._peek()
        if t in ("!", "~"):
            self._take()
            return 1 - self._unary()
        if t == "(":
            self._take()
            v = self._or()
            if self._take() != ")":
                raise SdfError("unbalanced condition")
            return v
        if t is None:
            raise SdfError("truncated condition")
        self._take()
        if "'" in t:
            return int(t[-1])
        if t in ("0", "1"):
            return int(t)
        if t not in self.env:
            raise SdfError("condition names %r, not one of the other pins" % t)
        return self.env[t]


# ---- values ----------------------------------------------------------------------

def _timescale(items):
    s = "".join(items)
    m = re.fullmatch(r"(1|10|100)(\.0*)?(s|ms|us|ns|ps|fs)", s)
    if not m:
        raise SdfError("bad TIMESCALE %r" % s)
    return int(m.group(1)) * _FS[m.group(3)]


def _value(item, file_fs, unit_fs):
    """One delay value list: [] -> INF, [v] or [min:typ:max] -> integer units."""
    if not isinstance(item, list):
        raise SdfError("delay value must be parenthesised: %r" % item)
    if len(item) == 0:
        return INF
    if len(item) != 1:
        raise SdfError("bad delay value %r" % item)
    parts = item[0].split(":")
    if len(parts) == 3:
        text = parts[1]
    elif len(parts) == 1:
        text = parts[0]
    else:
        raise SdfError("bad delay value %r" % item)
    x = Fraction(text) * file_fs / unit_fs
    if x < 0:
        raise SdfError("negative delay %s" % text)
    n = int(x + Fraction(1, 2))          # nearest integer, halves up
    if n >= INF:
        raise SdfError("delay %s too large" % text)
    return n


def _rise_fall(vals, file_fs, unit_fs):
    if len(vals) == 0:
        raise SdfError("IOPATH without delay values")
    r = _value(vals[0], file_fs, unit_fs)
    f = _value(vals[1], file_fs, unit_fs) if len(vals) > 1 else r
    return r, f


# ---- translation -----------------------------------------------------------------

def annotate(text, type_names, type_pins, gate_type, instance_names, fanin_off, gate_dly_off, dly_len, unit_fs,
             out_pin="Y"):
    """Delay tables (int32 [dly_len], laid out as the netlist's gate_dly_off says) and
    interconnect delays (int32 wire_rise [E], wire_fall [E]) from SDF text.

    type_pins[t] lists type t's input pin names in pin order; instance_names[g] is
    gate g's SDF instance; fanin_off[g] .. fanin_off[g+1]-1 are its fanin edges."""
    tree = _tree(text)
    if not tree or tree[0] != "DELAYFILE":
        raise SdfError("not a DELAYFILE")
    G = len(gate_type)
    E = int(fanin_off[G])
    inst_of = {name: g for g, name in enumerate(instance_names)}
    dly = np.zeros(int(dly_len), dtype=np.int64)
    wire_rise = np.zeros(E, dtype=np.int64)
    wire_fall = np.zeros(E, dtype=np.int64)
    file_fs = 10**6                      # SDF's default TIMESCALE, 1 ns
    for item in tree[1:]:
        if isinstance(item, list) and item and item[0] == "TIMESCALE":
            file_fs = _timescale(item[1:])
    tables = {}          # g -> [4n][cols] array, INF where nothing is set
    for g in range(G):
        n = len(type_pins[gate_type[g]])
        tables[g] = np.full((4 * n, 1 << (n - 1)), INF, dtype=np.int64)

    for cell in tree[1:]:
        if not (isinstance(cell, list) and cell and cell[0] == "CELL"):
            continue
        celltype, inst, stmts = None, None, []
        for part in cell[1:]:
            if part[0] == "CELLTYPE":
                celltype = part[1].strip('"')
            elif part[0] == "INSTANCE":
                inst = part[1] if len(part) > 1 else ""
            elif part[0] == "DELAY":
                for block in part[1:]:
                    if block[0] != "ABSOLUTE":
                        raise SdfError("only ABSOLUTE delays are read, not %s" % block[0])
                    stmts += block[1:]
        g = inst_of.get(inst) if inst else None
        if inst and g is None:
            raise SdfError("unknown instance %r" % inst)
        if g is not None and celltype != type_names[gate_type[g]]:
            raise SdfError("instance %s is a %s, not a %s" % (inst, type_names[gate_type[g]], celltype))
        conds = []
        for st in stmts:
            if st[0] == "INTERCONNECT":
                dst = st[2]
                if "/" not in dst:
                    raise SdfError("INTERCONNECT destination %r is not inst/pin" % dst)
                dinst, dpin = dst.rsplit("/", 1)
                if dinst not in inst_of:
                    raise SdfError("unknown instance %r" % dinst)
                dg = inst_of[dinst]
                pins = type_pins[gate_type[dg]]
                if dpin not in pins:
                    raise SdfError("%s has no pin %s" % (dinst, dpin))
                e = int(fanin_off[dg]) + list(pins).index(dpin)
                wire_rise[e], wire_fall[e] = _rise_fall(st[3:], file_fs, unit_fs)
            elif st[0] == "IOPATH":
                if g is None:
                    raise SdfError("IOPATH outside an instance")
                _iopath(tables[g], type_pins[gate_type[g]], out_pin, st, None, file_fs, unit_fs)
            elif st[0] == "COND":
                if g is None:
                    raise SdfError("COND outside an instance")
                conds.append(st)
            else:
                raise SdfError("unsupported statement %s" % st[0])
        for st in conds:             # after every unconditional statement, in file order
            body = st[-1]
            expr = st[1:-1]
            if expr and isinstance(expr[0], str) and expr[0].startswith('"'):
                expr = expr[1:]      # a condition name
            if not (isinstance(body, list) and body and body[0] == "IOPATH"):
                raise SdfError("COND without IOPATH")
            _iopath(tables[g], type_pins[gate_type[g]], out_pin, body, _Cond(_flatten(expr)), file_fs, unit_fs)

    for g in range(G):
        t = tables[g]
        dly[int(gate_dly_off[g]):int(gate_dly_off[g]) + t.size] = t.ravel()
    return dly.astype(np.int32), wire_rise.astype(np.int32), wire_fall.astype(np.int32)


def _iopath(table, pins, out_pin, st, cond, file_fs, unit_fs):
    port, out = st[1], st[2]
    if out != out_pin:
        raise SdfError("IOPATH to %r, not the output %r" % (out, out_pin))
    if isinstance(port, list):
        if len(port) != 2 or port[0] not in ("posedge", "negedge"):
            raise SdfError("bad port %r" % port)
        edges = [0] if port[0] == "posedge" else [1]
        name = port[1]
    else:
        edges, name = [0, 1], port
    if name not in pins:
        raise SdfError("no pin %r" % name)
    i = list(pins).index(name)
    n = len(pins)
    r, f = _rise_fall(st[3:], file_fs, unit_fs)
    others = [p for p in pins if p != name]
    if cond is not None and name in cond.names:
        raise SdfError("a condition names the switching pin %s" % name)
    for c in range(1 << (n - 1)):
        if cond is not None:
            env = {others[k]: (c >> (n - 2 - k)) & 1 for k in range(n - 1)}
            if not cond.value(env):
                continue
        for e_in in edges:
            table[4 * i + 2 * e_in + 0, c] = r
            table[4 * i + 2 * e_in + 1, c] = f
