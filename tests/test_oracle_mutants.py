"""Plant one plausible mistake at a time in a copy of oracle.c (on the CPU) and
check that the pins catch every one of them: a dropped term, a wrong sign or
identity, an off-by-one index, a transposed operand, inclusive/exclusive
confusion, a narrower accumulator."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "u32_add_exclusive_shifted": (
        "        if (!inclusive)\n            y[i] = acc;\n        acc = acc + xi;",
        "        acc = acc + xi;\n        if (!inclusive)\n            y[i] = acc;"),
    "u32_add_dropped_accumulator": ("        acc = acc + xi;\n        if (inclusive)\n            y[i] = acc;\n    }\n}\n\n/* Plain scan with u32 maximum",
                                    "        acc = xi;\n        if (inclusive)\n            y[i] = acc;\n    }\n}\n\n/* Plain scan with u32 maximum"),
    "u32_add_wrong_identity": ("uint32_t acc = 0u; /* additive identity */",
                               "uint32_t acc = 1u; /* additive identity */"),
    "u32_max_flipped_compare": ("acc = (xi > acc) ? xi : acc;", "acc = (xi < acc) ? xi : acc;"),
    "u32_max_transposed_select": ("acc = (xi > acc) ? xi : acc;", "acc = (xi > acc) ? acc : xi;"),
    "f32_abs_lost_sign": ("aacc = aacc + (xi < 0.0 ? -xi : xi);", "aacc = aacc + xi;"),
    "f32_float_accumulator": ("double acc = 0.0, aacc = 0.0;",
                              "float acc = 0.0f; double aacc = 0.0;"),
    "f32_exclusive_includes_self": ("            if (y) y[i] = acc;\n            if (absy) absy[i] = aacc;\n        }\n        acc",
                                    "            if (y) y[i] = acc + xi;\n            if (absy) absy[i] = aacc;\n        }\n        acc"),
    "segmented_start_off_by_one": ("uint64_t lo = offsets[s], hi = offsets[s + 1];",
                                   "uint64_t lo = offsets[s] ? offsets[s] - 1 : 0, hi = offsets[s + 1];"),
    "segmented_end_off_by_one": ("uint64_t lo = offsets[s], hi = offsets[s + 1];",
                                 "uint64_t lo = offsets[s], hi = offsets[s + 1] + 1;"),
    "segmented_transposed_bounds": ("uint64_t lo = offsets[s], hi = offsets[s + 1];",
                                    "uint64_t lo = offsets[s + 1], hi = offsets[s];"),
    "segmented_no_reset": ("        uint32_t acc = 0u;\n        for (uint64_t i = lo; i < hi; ++i) {",
                           "        static uint32_t acc;\n        for (uint64_t i = lo; i < hi; ++i) {"),
    "compact_inverted_flag": ("if (flags[i] != 0) {", "if (flags[i] == 0) {"),
    "compact_wrong_source_index": ("src + i * record_bytes", "src + (i ? i - 1 : 0) * record_bytes"),
    "compact_count_dropped": ("            ++k;\n", "            k = 1;\n"),
    "reduce_start_off_by_one": ("        uint32_t acc = 0u;\n        for (uint64_t i = first; i < end; ++i)\n            acc = acc + values[i];",
                                "        uint32_t acc = 0u;\n        for (uint64_t i = first + 1; i < end; ++i)\n            acc = acc + values[i];"),
    "reduce_end_inclusive": ("        uint32_t acc = 0u;\n        for (uint64_t i = first; i < end; ++i)\n            acc = acc + values[i];",
                             "        uint32_t acc = 0u;\n        for (uint64_t i = first; i <= end && i < n; ++i)\n            acc = acc + values[i];"),
    "reduce_no_reset": ("        uint32_t acc = 0u;\n        for (uint64_t i = first; i < end; ++i)\n            acc = acc + values[i];",
                        "        static uint32_t acc;\n        for (uint64_t i = first; i < end; ++i)\n            acc = acc + values[i];"),
    "reduce_wrong_slot": ("        out[s] = acc;", "        out[s ? s - 1 : 0] = acc;"),
    "recurrence_a_index_shifted": ("double at = (double)a[t], bt = (double)b[t];",
                                   "double at = (double)a[t ? t - 1 : 0], bt = (double)b[t];"),
    "recurrence_initial_state_one": ("double h = 0.0, g = 0.0;", "double h = 1.0, g = 0.0;"),
    "recurrence_roles_swapped": ("h = at * h + bt;", "h = bt * h + at;"),
    "recurrence_dropped_coefficient": ("h = at * h + bt;", "h = h + bt;"),
    "recurrence_magnitude_lost_abs": ("g = (at < 0.0 ? -at : at) * g + (bt < 0.0 ? -bt : bt);",
                                      "g = at * g + bt;"),
    "recurrence_exclusive_after_step": ("        if (!inclusive) {\n            if (y) y[t] = h;",
                                        "        if (!inclusive) {\n            if (y) y[t] = at * h + bt;"),
    "recurrence_float_state": ("double h = 0.0, g = 0.0;", "float h = 0.0f; double g = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor must be unique: " + name
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(mutated), str(tmp_path / "liboracle_mutant.so"), force=True))
    o = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, "no pin caught mutant " + name
