"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle.c (on the CPU, in a temporary
directory), builds it, and runs the pin tests against that build in a child
process (ORACLE_LIB).  Every mutant must make at least one pin fail.
Mistakes that would read or write outside the test buffers are not planted.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "swizzle_shift_4": ("const int32_t S = 3;", "const int32_t S = 4;"),
    "swizzle_chunk_bits_3": ("const int32_t M = 4;", "const int32_t M = 3;"),
    "swizzle_or_not_xor": ("return offset ^ ((offset & source_mask) >> S);",
                           "return offset | ((offset & source_mask) >> S);"),
    "box_bytes_without_element_size": ("return elems * (uint64_t)v->esize;", "return elems;"),
    "grid_y_fastest": ("for (int32_t d = 0; d < v->rank; ++d) {\n            uint64_t n_d",
                       "for (int32_t d = v->rank - 1; d >= 0; --d) {\n            uint64_t n_d"),
    "oob_fill_ff": ("= inside ? base[addr + (uint64_t)b] : 0;", "= inside ? base[addr + (uint64_t)b] : 0xFF;"),
    "lower_bound_off_by_one": ("if (g[d] < 0 || g[d] >= (int64_t)v->dims[d]) inside = 0;",
                               "if (g[d] < 1 || g[d] >= (int64_t)v->dims[d]) inside = 0;"),
    "upper_bound_off_by_one": ("if (g[d] < 0 || g[d] >= (int64_t)v->dims[d]) inside = 0;",
                               "if (g[d] < 0 || g[d] >= (int64_t)v->dims[d] - 1) inside = 0;"),
    "traversal_step_ignored": ("g[d] = (int64_t)c[d] + k * (int64_t)step_along(v, d);", "g[d] = (int64_t)c[d] + k;"),
    "store_unswizzled": ("base[addr + (uint64_t)b] = image[oracle_swizzle(o, v->swizzle_bits)];",
                         "base[addr + (uint64_t)b] = image[o];"),
    "oob_mask_unswizzled": ("image[oracle_swizzle(o, v->swizzle_bits)] = outside;", "image[o] = outside;"),
    "oob_mask_inverted": ("uint8_t outside = element_in_bounds(v, c, e, g) ? 0 : 1;",
                          "uint8_t outside = element_in_bounds(v, c, e, g) ? 1 : 0;"),
    "roundtrip_stores_through_source_view": ("    oracle_tile_store(dst, dst_base, coords, n, packed);\n    free(packed);\n    return 0;\n}\n\n/*",
                                             "    oracle_tile_store(src, dst_base, coords, n, packed);\n    free(packed);\n    return 0;\n}\n\n/*"),
    "add_subtracts": ("x = x + addend;", "x = x - addend;"),
    "roundtrip_skips_store": ("    oracle_tile_store(dst, dst_base, coords, n, packed);\n    free(packed);\n    return 0;\n}\n\n/*",
                              "    free(packed);\n    return 0;\n}\n\n/*"),
    "grid_drops_ragged_last_tile": ("return (v->dims[d] + v->box[d] - 1) / v->box[d];", "return v->dims[d] / v->box[d];"),
    "visits_rounded_down": ("return (v->box[d] + step_along(v, d) - 1) / step_along(v, d);",
                            "return v->box[d] / step_along(v, d);"),
    "grid_origin_is_tile_index": ("= (int32_t)(t_d * v->box[d]);", "= (int32_t)t_d;"),
    "address_without_strides": ("addr += (uint64_t)g[d] * v->strides[d];", "addr += (uint64_t)g[d] * (uint64_t)v->esize;"),
    "load_forgets_fill": ("= inside ? base[addr + (uint64_t)b] : 0;", "= base[addr + (uint64_t)b];"),
    "packed_slots_by_elements": ("uint8_t* image = packed + i * box_bytes;", "uint8_t* image = packed + i * box_elems;"),
    "box_index_split_by_extent_not_visits": ("int64_t k = (int64_t)(rest % visits_along(v, d));\n        rest /= visits_along(v, d);",
                                             "int64_t k = (int64_t)(rest % v->box[d]);\n        rest /= v->box[d];"),
    "store_in_reverse_list_order": ("for (uint64_t i = 0; i < n; ++i) {\n        const int32_t* c = coords + i * (uint64_t)v->rank;\n        const uint8_t* image",
                                    "for (uint64_t i = n; i-- > 0;) {\n        const int32_t* c = coords + i * (uint64_t)v->rank;\n        const uint8_t* image"),
    "update_skipped": ("    oracle_add_f32(packed, n * box_bytes, addend);\n", ""),
    "update_first_box_only": ("oracle_add_f32(packed, n * box_bytes, addend);", "oracle_add_f32(packed, box_bytes, addend);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(before, after, 1)
    c_path = tmp_path / "oracle.c"
    c_path.write_text(mutated)
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib),
                           str(c_path)])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout or "Error" in r.stdout
