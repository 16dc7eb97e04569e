"""Parity of the library's SDF translator (gatspi_sdf_annotate, host code behind the C
ABI) with the oracle's translation: identical tables and wire delays on the hand-
worked statements, on synthetic SDF of many netlists, spellings and time scales,
and the same refusals.  The translator uses no GPU; the last test simulates on the
GPU from translated tables.
"""
import numpy as np
import pytest

import synth
import test_oracle_sdf as ts
from oracle import sdf as osdf


class _Lib:
    """The library's translator with the oracle's calling convention."""

    class SdfError(Exception):
        pass

    @staticmethod
    def annotate(text, type_names, type_pins, gate_type, instance_names, fanin_off, gate_dly_off, dly_len, unit_fs):
        from gate_level_logic_gb300 import GatspiError, sdf_annotate
        try:
            return sdf_annotate(text, type_names, type_pins, gate_type, instance_names, fanin_off, gate_dly_off,
                                dly_len, unit_fs)
        except GatspiError as e:
            assert e.name == "GATSPI_EINVAL", e
            raise _Lib.SdfError(str(e))


@pytest.fixture(scope="module")
def lib():
    from gate_level_logic_gb300 import build
    build.build()
    return _Lib


@pytest.mark.parametrize("name", sorted(ts.HAND))
def test_hand_statements(lib, name):
    text, cells, _ = ts.HAND[name]
    got = ts.translate(lib, text, cells)
    want = ts.translate(osdf, text, cells)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


def test_fig4_and_interconnect(lib):
    ts.test_fig4_aoi21(lib)
    ts.test_interconnect(lib)


@pytest.mark.parametrize("name", sorted(ts.ERRORS))
def test_same_refusals(lib, name):
    with pytest.raises(lib.SdfError):
        ts.translate(lib, ts.ERRORS[name], ts.NAND2)


@pytest.mark.parametrize("seed", range(12))
def test_synthetic_netlists(lib, seed):
    rng = np.random.default_rng(seed)
    net = synth.generate_netlist(synth.NetlistSpec(
        num_gates=int(rng.integers(50, 2000)), num_inputs=int(rng.integers(2, 40)), num_levels=int(rng.integers(1, 8)),
        seed=seed, cell_mix=[synth.CELL_MIX, ("random", 2), ("random", 4), ("random", 1)][seed % 4],
        cond_cells=("AOI21", "MUX2", "OAI22", "NAND4"), cond_fraction=float(rng.choice([0.0, 0.5, 1.0])),
        delay_mode=("arc", "pin_out")[seed % 2], wire_delay=(0, int(rng.integers(0, 50)))))
    unit = ["1ps", "1ns", "10ps", "100ps"][seed % 4]
    s = synth.write_sdf(net, seed=seed, file_unit=unit)
    args = (s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names, net.fanin_off, net.gate_dly_off,
            net.dly_data.size, 1000)
    got = lib.annotate(*args)
    want = osdf.annotate(*args)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
    assert np.array_equal(got[0], net.dly_data)


def test_coarser_simulation_unit_rounds_like_the_oracle(lib):
    """The tables in 1 ps, translated into a 10 ps simulator unit: every value rounds."""
    net, _ = synth.make("tiny")
    s = synth.write_sdf(net, seed=7, file_unit="1ps")
    args = (s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names, net.fanin_off, net.gate_dly_off,
            net.dly_data.size, 10000)
    got, want = lib.annotate(*args), osdf.annotate(*args)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
    finite = net.dly_data != synth.INF
    assert np.array_equal(got[0][finite], (net.dly_data[finite] + 5) // 10)


@pytest.mark.gpu
def test_simulation_from_translated_tables(lib, oracle_lib):
    """The 50k workload's delays written as SDF, translated by the library and
    simulated on the GPU, equal the oracle simulating the oracle's translation."""
    import copy
    from test_gpu_parity import assert_same, pool_for, run_gpu
    from gate_level_logic_gb300 import Simulator
    net, stim = synth.make("50k")
    s = synth.write_sdf(net, seed=11, file_unit="1ns")
    args = (s.text, net.type_names, s.pin_names, net.gate_type, s.instance_names, net.fanin_off, net.gate_dly_off,
            net.dly_data.size, 1000)
    mine, theirs = copy.copy(net), copy.copy(net)
    mine.dly_data, mine.wire_rise, mine.wire_fall = lib.annotate(*args)
    theirs.dly_data, theirs.wire_rise, theirs.wire_fall = osdf.annotate(*args)
    ref = oracle_lib.simulate(theirs, stim, threads=8)
    assert_same(run_gpu(Simulator, mine, stim, pool_for(ref, mine)), ref, "from SDF")


def _nested_condition(levels):
    """B || B && B | B ^ B & B == (...): each level leaves six operands pending, one per
    binary precedence level, and nests one parenthesis deeper."""
    s = "B"
    for _ in range(levels):
        s = "B || B && B | B ^ B & B == (%s)" % s
    return s


def test_condition_operand_bound(lib):
    """A condition whose evaluation would hold more operands at once than the
    translator's evaluation stack (256) is refused, though its nesting is within the
    limit; one within the bound translates as the oracle translates it."""
    text = ts._wrap(ts._cell("(COND %s (IOPATH (posedge A) Y (1)))" % _nested_condition(45)))
    with pytest.raises(lib.SdfError, match="too long"):
        ts.translate(lib, text, ts.NAND2)
    text = ts._wrap(ts._cell("(COND %s (IOPATH (posedge A) Y (3)))" % _nested_condition(20)))
    for a, b in zip(ts.translate(lib, text, ts.NAND2), ts.translate(osdf, text, ts.NAND2)):
        assert np.array_equal(a, b)


def test_deeply_nested_lists_are_refused(lib):
    """SDF lists nested 100000 deep (inside a COND) are refused with EINVAL when the
    text is parsed, before anything walks them recursively."""
    deep = "(" * 100000 + "B" + ")" * 100000
    text = ts._wrap(ts._cell("(COND %s (IOPATH (posedge A) Y (1)))" % deep))
    with pytest.raises(lib.SdfError, match="nested too deeply"):
        ts.translate(lib, text, ts.NAND2)


def test_number_precision_bound(lib):
    """Delay values keep 20 significant digits exactly, and zeros after them, whatever
    the TIMESCALE (up to 100 s, where 20 digits times the file unit still fit the
    translator's 128-bit arithmetic) and however small (a value below half a unit is
    0, exactly half rounds up); a value with more significant digits is refused, never
    rounded off and never overflowed."""
    cases = (("1.00000000000000000000000000", "1ns"),       # zeros beyond 20 digits: exact
             ("0.12345678901234567890", "1ns"),             # 20 digits: 123 ps
             ("3.1400000000000000000000000000", "1ps"),     # 3 ps
             ("99999999999999999999", "100s"),              # the largest mantissa and file unit: too large
             (".721812064E-24", "100ns"),                   # far below one unit: 0, exactly
             ("5e-4", "1ns"),                                # exactly one half a unit: rounds up to 1
             ("4.9999999999999999999e-4", "1ns"))           # just below one half: 0
    for value, unit in cases:
        text = ts._wrap(ts._cell("(IOPATH A Y (%s))" % value), timescale="(TIMESCALE %s)" % unit)
        try:
            want = ts.translate(osdf, text, ts.NAND2)
        except osdf.SdfError:
            with pytest.raises(lib.SdfError, match="too large"):
                ts.translate(lib, text, ts.NAND2)
            continue
        for a, b in zip(ts.translate(lib, text, ts.NAND2), want):
            assert np.array_equal(a, b), value
    for value in ("1.000000000000000000001", "123456789012345678901", "9" * 29):
        text = ts._wrap(ts._cell("(IOPATH A Y (%s))" % value), timescale="(TIMESCALE 100s)")
        with pytest.raises(lib.SdfError, match="significant digits"):
            ts.translate(lib, text, ts.NAND2)


@pytest.mark.parametrize("lit", ["1'1", "1'bc0", "1'b10", "'1", "1'x1", "a'b1"])
def test_malformed_literals_are_refused_by_both(lib, lit):
    """Only one-bit binary literals are conditions' constants (0, 1, 1'b0, 1'b1, 'b0,
    'b1, any size digits): anything else with a quote is refused, by the library as by
    the oracle."""
    text = ts._wrap(ts._cell("(COND B == %s (IOPATH (posedge A) Y (1)))" % lit))
    with pytest.raises(osdf.SdfError):
        ts.translate(osdf, text, ts.NAND2)
    with pytest.raises(lib.SdfError):
        ts.translate(lib, text, ts.NAND2)


@pytest.mark.parametrize("lit", ["1'b1", "1'B0", "'b1", "4'b0", "0", "1"])
def test_literals_translate_like_the_oracle(lib, lit):
    text = ts._wrap(ts._cell("(COND B == %s (IOPATH (posedge A) Y (2)))" % lit))
    for a, b in zip(ts.translate(lib, text, ts.NAND2), ts.translate(osdf, text, ts.NAND2)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("spelling", ['NAND2"', '"NAND2""'])
def test_celltype_quotes_as_the_oracle_reads_them(lib, spelling):
    """A CELLTYPE with a stray quote (found by a differential fuzz): the library reads
    the name as the oracle does, without every quote around it, and both then agree
    (or both refuse)."""
    text = ts._wrap(ts._cell("(IOPATH A Y (1))")).replace('(CELLTYPE "NAND2")', "(CELLTYPE %s)" % spelling)
    assert spelling in text
    try:
        want = ts.translate(osdf, text, ts.NAND2)
    except osdf.SdfError:
        with pytest.raises(lib.SdfError):
            ts.translate(lib, text, ts.NAND2)
        return
    for a, b in zip(ts.translate(lib, text, ts.NAND2), want):
        assert np.array_equal(a, b)


def _random_conditions(rng):
    """One cell's statements: up to four COND IOPATHs, each with a random well-formed
    condition over the other three pins (every operator, literal form, optional
    parentheses and spacing), and sometimes an unconditional IOPATH."""
    pins = ("A", "B", "C", "D")
    lits = ["0", "1", "1'b0", "1'b1", "'b0", "'b1", "1'B1", "4'b0"]
    ops = ["&", "|", "^", "&&", "||", "==", "===", "!=", "!=="]

    def space():
        return rng.choice(["", " ", "  "])

    def expr(depth, others):
        r = rng.random()
        if depth <= 0 or r < 0.3:
            return rng.choice(others) if rng.random() < 0.75 else rng.choice(lits)
        if r < 0.45:
            inner = expr(depth - 1, others)
            return rng.choice(["!", "~"]) + space() + "(" + inner + ")"
        left, right = expr(depth - 1, others), expr(depth - 1, others)
        if rng.random() < 0.3:
            left = "(" + left + ")"
        return left + space() + rng.choice(ops) + space() + right

    stmts = []
    for _ in range(rng.randint(1, 4)):
        sw = rng.choice(pins)
        others = [p for p in pins if p != sw]
        edge = rng.choice(["(posedge %s)" % sw, "(negedge %s)" % sw, sw])
        stmts.append("(COND %s (IOPATH %s Y (%d) (%d)))"
                     % (expr(rng.randint(1, 6), others), edge, rng.randint(1, 50), rng.randint(1, 50)))
    if rng.random() < 0.5:
        stmts.insert(0, "(IOPATH A Y (60) (61))")
    return " ".join(stmts)


def test_random_conditions_translate_like_the_oracle(lib):
    """400 seeded random condition sets on a four-pin cell: the library's tables equal
    the oracle's (precedence, ===, !==, ~, ^, sized and unsized literals)."""
    import random
    rng = random.Random(2027)
    cells = [("u", "NAND4", ("A", "B", "C", "D"))]
    for k in range(400):
        text = ts._wrap(ts._cell(_random_conditions(rng), tname="NAND4"))
        for a, b in zip(ts.translate(lib, text, cells), ts.translate(osdf, text, cells)):
            assert np.array_equal(a, b), (k, text)
