"""The oracle pins must catch plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake by a textual
substitution (a wrong shift, a dropped term, a swapped nibble, an off-by-one
index, a wrong tie-break ...), compiles the copy to a temporary library and runs
the pin battery of ``test_oracle_pins`` against it in a child process. The case
passes only if the battery fails. Everything runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
E5M2_MARKER = "/* ====================================================== FP8 E5M2 variant"

MUTANTS = {
    "exponent shift": ("return (uint8_t)((x >> 7) & 0xFF);", "return (uint8_t)((x >> 8) & 0xFF);"),
    "sign bit dropped from a": ("(uint8_t)(((x >> 8) & 0x80) | (x & 0x7F))", "(uint8_t)((x & 0x7F))"),
    "mantissa mask in rebuild": ("(unsigned)(a & 0x7F));", "(unsigned)(a & 0x3F));"),
    "tie-break reversed": ("hist[order[j]] < hist[v]", "hist[order[j]] <= hist[v]"),
    "histogram bin index": ("hist[exponent_of(x[i])]++", "hist[exponent_of(x[i]) & 0x7F]++"),
    "dummy code not 0": ("enc[v] = 0;", "enc[v] = 15;"),
    "nibble order in encode": ("B[i / 2] = code;", "B[i / 2] = (uint8_t)(code << 4);"),
    "nibble order in decode": ("(B[i / 2] >> (4 * (i % 2)))", "(B[i / 2] >> (4 * ((i + 1) % 2)))"),
    "position not chunk-relative": ("(uint32_t)(i - start));", "(uint32_t)(i));"),
    "inclusive offsets": ("put_u32(C + 4 * c, (uint32_t)running);", "put_u32(C + 4 * c, (uint32_t)(running + k));"),
    "values not after positions": ("block[2 * k + j] = e;", "block[k + j] = e;"),
    "escape fix-up dropped": ("x[start + pos] = rebuild(A[start + pos], block[2 * k + j]);",
                              "x[start + pos] = x[start + pos];"),
    "section padding": ("return (v + 15) / 16 * 16;", "return (v + 7) / 8 * 8;"),
    "chunk count": ("L.nc = (n + chunk - 1) / chunk;", "L.nc = n / chunk + 1;"),
    "first offset not checked": ("if (get_u32(C) != 0 || get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;",
                                 "if (get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;"),
    "last offset not checked": ("if (get_u32(C) != 0 || get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;",
                                "if (get_u32(C) != 0) return ORC_ERR_CORRUPT;"),
    "repeated positions accepted": ("if (j > 0 && pos <= get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;",
                                    "if (j > 0 && pos < get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;"),
    "falling positions accepted": ("if (j > 0 && pos <= get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;",
                                   "if (j > 0 && pos == get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;"),
}

BATTERY = r"""
import sys, importlib.util
sys.path.insert(0, {root!r}); sys.path.insert(0, {here!r})
import oracle
spec = importlib.util.spec_from_file_location("pins", {pins!r})
pins = importlib.util.module_from_spec(spec); spec.loader.exec_module(pins)
o = oracle.Oracle(oracle.load({lib!r}))
checks = [
    lambda: pins.test_split_hand_worked_examples(o),
    lambda: pins.test_split_matches_ieee_fields_exhaustively(o),
    lambda: pins.test_merge_is_a_bijection_inverse_of_split(o),
    lambda: pins.test_histogram_is_bincount_of_ieee_exponents(o),
    lambda: pins.test_top16_hand_built(o, [(200, 5), (100, 7), (7, 5)],
                                       [100, 7, 200, 0, 1, 2, 3, 4, 5, 6, 8, 9, 10, 11, 12, 13]),
    lambda: pins.test_luts_are_consistent_with_codebook(o),
    lambda: pins.test_encode_matches_hand_worked_stream(o),
    lambda: pins.test_brute_force_tiny_inputs(o, 24),
    lambda: pins.test_brute_force_tiny_inputs(o, 1024),
    lambda: pins.test_all_patterns_tensor(o),
    lambda: pins.test_all_zero_reaches_four_thirds(o),
    lambda: pins.test_decode_rejects_corrupt_streams(o),
]
failed = []
for i, c in enumerate(checks):
    try:
        c()
    except Exception as ex:  # an assertion or a parse error of a malformed stream
        failed.append((i, type(ex).__name__))
print("FAILED", failed)
sys.exit(1 if failed else 0)
"""


def _run_battery(lib_path):
    code = BATTERY.format(root=os.path.dirname(HERE), here=HERE, lib=lib_path,
                          pins=os.path.join(HERE, "test_oracle_pins.py"))
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)


def test_battery_passes_on_the_real_oracle():
    r = _run_battery(oracle.build())
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "uzip_oracle.c")).read()
    head, tail = src.split(E5M2_MARKER, 1)  # the BF16 part, then the E5M2 variant
    assert head.count(old) == 1, f"mutation site for {name!r} not unique"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(head.replace(old, new) + E5M2_MARKER + tail)
    lib = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / "libmutant.so"))
    r = _run_battery(lib)
    assert r.returncode != 0, f"mutant {name!r} survived the pins:\n{r.stdout}{r.stderr}"
