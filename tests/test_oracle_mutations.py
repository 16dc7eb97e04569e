"""The oracle's pins are sharp: each plausible slip planted in a copy of the oracle
source (compiled on the CPU, in a temporary directory) fails at least one pin.

The committed oracle is never modified; every mutant is a text substitution applied
to a temporary copy.
"""
import functools
import os
import shutil
import types

import pytest

import oracle
import test_oracle_golden as golden
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__))

MUTANTS = {
    "wire filter tested once, not repeated": (
        "if (g_literal_skip && skipped) break;", "if (skipped) break;"),
    "wire filter not strict": (
        "(int64_t)Win[i][p[i] + 1] < 0)", "(int64_t)Win[i][p[i] + 1] <= 0)"),
    "wire rise/fall swapped": (
        "d = (p[i] % 2) ? wire_fall[i] : wire_rise[i];", "d = (p[i] % 2) ? wire_rise[i] : wire_fall[i];"),
    "gate filter not strict": (
        "if (t_o - (int64_t)O->w[po] < reject_limit(d, q)) {",
        "if (t_o - (int64_t)O->w[po] <= reject_limit(d, q)) {"),
    "gate filter never cancels": (
        "if (t_o - (int64_t)O->w[po] < reject_limit(d, q)) {", "if (0) {"),
    "wire filter ignores PATHPULSEPERCENT": (
        "reject_limit(d, q) - (int64_t)Win[i][p[i] + 1] < 0)", "d - (int64_t)Win[i][p[i] + 1] < 0)"),
    "gate filter ignores PATHPULSEPERCENT": (
        "if (t_o - (int64_t)O->w[po] < reject_limit(d, q)) {", "if (t_o - (int64_t)O->w[po] < d) {"),
    "reject limit rounded up": (
        "return d * q / 100;", "return (d * q + 99) / 100;"),
    "a cancel never exposes a pending entry": (
        "if (t_o - (int64_t)O->w[po] < reject_limit(d, q)) {",
        "if (t_o - (int64_t)O->w[po] < reject_limit(d, q) && (po < 1 || O->w[po - 1] <= t)) {"),
    "MSI takes the last finite arc, not the smallest": (
        "if (dd != NO_ARC && dd < d) d = dd;", "if (dd != NO_ARC) d = dd;"),
    "row: input and output edge transposed": (
        "const int64_t row = 4 * i + 2 * e_in + e_out;", "const int64_t row = 4 * i + 2 * e_out + e_in;"),
    "input edge sense flipped": (
        "const int e_in = (p[i] % 2) ? RISE : FALL;", "const int e_in = (p[i] % 2) ? FALL : RISE;"),
    "column with the first pin least significant": (
        "if (j != i) col = col * 2 + (p[j] % 2);",
        "if (j != i) col += (int64_t)(p[j] % 2) << (j < i ? j : j - 1);"),
    "column from values before the switch": (
        "if (j != i) col = col * 2 + (p[j] % 2);", "if (j != i) col = col * 2 + ((p[j] - sw[j]) % 2);"),
    "only one simultaneous pin switches": (
        "            sw[i] = (a[i] == t);\n            if (sw[i]) p[i] += 1;",
        "            sw[i] = (a[i] == t);\n            for (int j = 0; j < i; ++j) if (sw[j]) sw[i] = 0;\n"
        "            if (sw[i]) p[i] += 1;"),
    "initial value ignored": (
        "p[i] = (Win[i][0] == -1) ? 1 : 0;", "p[i] = 0;"),
    "toggle count includes the head": (
        "*tc = po - (y0 ? 1 : 0);", "*tc = po;"),
    "time at 1 clipped one unit short": (
        "if (e > Lw) e = Lw;", "if (e > Lw - 1) e = Lw - 1;"),
    "time at 1 counts the value-0 intervals": (
        "for (int64_t k = 1; k <= po; k += 2) {", "for (int64_t k = 0; k <= po; k += 2) {"),
}


def _battery(lib_path):
    """Run a compact set of pins through the oracle at lib_path; True if all hold."""
    shim = types.SimpleNamespace(simulate=functools.partial(oracle.simulate, lib_path=lib_path),
                                 bruteforce=functools.partial(oracle.bruteforce, lib_path=lib_path),
                                 OracleError=oracle.OracleError)
    checks = [
        lambda: golden.test_fig3_format_through_buffer_and_inverter(shim),
        lambda: golden.test_fig4_nand2_index_and_value(shim),
        lambda: golden.test_msi_takes_smallest_switching_arc(shim),
        lambda: golden.test_msi_skips_impossible_arc(shim),
    ]
    for a1, a2, e in [(0, 1, [-1, 0, 105, 307]), (0, 0, [-1, 0, 106, 308]), (1, 1, [0])]:
        checks.append(functools.partial(golden.test_fig4_aoi21_conditional_delay, shim, a1, a2, e))
    for seed in range(3):
        checks.append(functools.partial(pins.test_buffer_inverter_chain_is_inertial_delay_line, shim, seed))
    checks.append(lambda: pins.test_output_invariants(shim, "tiny"))

    for q in (50, 0):
        checks.append(functools.partial(golden.test_pulse_percent_worked_example, shim, q))
        checks.append(functools.partial(golden.test_pulse_percent_skewed_delays, shim, q))
        checks.append(functools.partial(pins.test_chain_with_pulse_limit_is_filtered_delay_line, shim, q, 0))

    def brute():
        import numpy as np
        for seed in range(150):
            net, stim = pins._random_case(seed)
            r = shim.simulate(net, stim)
            b = shim.bruteforce(net, stim)
            assert np.array_equal(r.pool, b.pool) and np.array_equal(r.tc, b.tc) and np.array_equal(r.t1, b.t1)
        for seed in range(100):
            net, stim = pins._random_case(seed)
            net = pins._skew_free(net)
            q = (0, 30, 50, 90)[seed % 4]
            r = shim.simulate(net, stim, pulse_percent=q)
            b = shim.bruteforce(net, stim, pulse_percent=q)
            assert np.array_equal(r.pool, b.pool) and np.array_equal(r.tc, b.tc) and np.array_equal(r.t1, b.t1)
    checks.append(brute)
    for c in checks:
        try:
            c()
        except (AssertionError, oracle.OracleError):
            return False
    return True


def _build_variant(tmp_path, old, new, target="gatspi_oracle.c"):
    d = tmp_path / "src"
    d.mkdir()
    for f in ("gatspi_oracle.c", "bruteforce.c", "testbench.c", "oracle_abi.h"):
        shutil.copy(os.path.join(SRC, f), d / f)
    text = (d / target).read_text()
    if old is not None:
        assert text.count(old) == 1, "mutation anchor not found exactly once: %r" % old
        text = text.replace(old, new)
    (d / target).write_text(text)
    return oracle.build(force=True, src_dir=str(d), out=str(tmp_path / "libvariant.so"))


def test_unmutated_copy_passes(tmp_path):
    assert _battery(_build_variant(tmp_path, None, None))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert not _battery(_build_variant(tmp_path, old, new)), "pins missed: " + name


# ---- the testbench restructuring (oracle/testbench.c) ----

TB_MUTANTS = {
    "boundary transition kept in the earlier window": (
        "while (!bad && x[i] != TB_EOW && x[i] < end) {", "while (!bad && x[i] != TB_EOW && x[i] <= end) {"),
    "boundary transition not folded into the initial value": (
        "while (x[i] != TB_EOW && x[i] <= start) {", "while (x[i] != TB_EOW && x[i] < start) {"),
    "times not made window-relative": (
        "bad = tb_push(&out, (int32_t)(x[i] - start));", "bad = tb_push(&out, (int32_t)x[i]);"),
    "window head written for the opposite value": (
        "int bad = value ? (tb_push(&out, -1) || tb_push(&out, 0)) : tb_push(&out, 0);",
        "int bad = !value ? (tb_push(&out, -1) || tb_push(&out, 0)) : tb_push(&out, 0);"),
    "every window starts from the testbench's initial value": (
        "        int64_t start = 0;\n        for (int32_t w = 0; w < W; ++w) {\n",
        "        int64_t start = 0;\n        for (int32_t w = 0; w < W; ++w) {\n            value = (x[0] == -1);\n"),
}


def _tb_battery(lib_path):
    import test_oracle_testbench as tbt
    shim = types.SimpleNamespace(restructure=functools.partial(oracle.restructure, lib_path=lib_path),
                                 OracleError=oracle.OracleError)
    checks = [lambda: tbt.test_restructure_equals_generator_windows(shim),
              lambda: tbt.test_boundary_transitions_fold_into_the_later_window(shim),
              lambda: tbt.test_initial_one_and_quiet_windows(shim),
              lambda: tbt.test_uneven_windows(shim),
              lambda: tbt.test_single_window_is_identity(shim)]
    checks += [functools.partial(tbt.test_windows_put_back_give_the_testbench, shim, seed) for seed in range(3)]
    for c in checks:
        try:
            c()
        except (AssertionError, oracle.OracleError):
            return False
    return True


def test_unmutated_testbench_copy_passes(tmp_path):
    assert _tb_battery(_build_variant(tmp_path, None, None, "testbench.c"))


@pytest.mark.parametrize("name", sorted(TB_MUTANTS))
def test_testbench_mutant_is_caught(tmp_path, name):
    old, new = TB_MUTANTS[name]
    assert not _tb_battery(_build_variant(tmp_path, old, new, "testbench.c")), "pins missed: " + name


# ---- the SDF translation (oracle/sdf.py) ----

SDF_MUTANTS = {
    "rise and fall swapped": (
        "            table[4 * i + 2 * e_in + 0, c] = r\n            table[4 * i + 2 * e_in + 1, c] = f",
        "            table[4 * i + 2 * e_in + 0, c] = f\n            table[4 * i + 2 * e_in + 1, c] = r"),
    "posedge read as the falling input edge": (
        'edges = [0] if port[0] == "posedge" else [1]', 'edges = [1] if port[0] == "posedge" else [0]'),
    "column with the first other pin least significant": (
        "env = {others[k]: (c >> (n - 2 - k)) & 1 for k in range(n - 1)}",
        "env = {others[k]: (c >> k) & 1 for k in range(n - 1)}"),
    "COND applied where it is written": (
        "                conds.append(st)",
        "                _iopath(tables[g], type_pins[gate_type[g]], out_pin, st[-1], _Cond(_flatten(st[1:-1])),"
        " file_fs, unit_fs)"),
    "first COND wins": ("        for st in conds:", "        for st in reversed(conds):"),
    "triple gives min": ("        text = parts[1]", "        text = parts[0]"),
    "rounding down": ("    n = int(x + Fraction(1, 2))", "    n = int(x)"),
    "one value leaves no fall delay": (
        "    f = _value(vals[1], file_fs, unit_fs) if len(vals) > 1 else r",
        "    f = _value(vals[1], file_fs, unit_fs) if len(vals) > 1 else INF"),
}


def _sdf_variant(tmp_path, old, new):
    import importlib.util
    text = open(os.path.join(SRC, "sdf.py")).read()
    if old is not None:
        assert text.count(old) == 1, "mutation anchor not found exactly once: %r" % old
        text = text.replace(old, new)
    path = tmp_path / "sdf_variant.py"
    path.write_text(text)
    spec = importlib.util.spec_from_file_location("sdf_variant_%d" % abs(hash(str(tmp_path))), path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _sdf_battery(mod):
    import test_oracle_sdf as ts
    checks = [lambda: ts.test_fig4_aoi21(mod), lambda: ts.test_interconnect(mod),
              lambda: ts.test_round_trip_tiny(mod, "1ns")]
    checks += [functools.partial(ts.test_hand_statements, mod, name) for name in sorted(ts.HAND)]
    checks += [functools.partial(ts.test_round_trip_conditional_cells, mod, seed) for seed in (0, 1)]
    for c in checks:
        try:
            c()
        except (AssertionError, mod.SdfError):
            return False
    return True


def test_unmutated_sdf_copy_passes(tmp_path):
    assert _sdf_battery(_sdf_variant(tmp_path, None, None))


@pytest.mark.parametrize("name", sorted(SDF_MUTANTS))
def test_sdf_mutant_is_caught(tmp_path, name):
    old, new = SDF_MUTANTS[name]
    assert not _sdf_battery(_sdf_variant(tmp_path, old, new)), "pins missed: " + name
