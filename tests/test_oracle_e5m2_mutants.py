"""The E5M2 pins must catch plausible mistakes in the oracle's E5M2 variant.

As for the BF16 part: each case plants one mistake in a copy of the oracle's
C source (inside its E5M2 part only), compiles it and runs the E5M2 pin
battery of ``test_oracle_e5m2_pins`` in a child process; the case passes only
if the battery fails. CPU only.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
E5M2_MARKER = "/* ====================================================== FP8 E5M2 variant"
SENTINEL_MARKER = "/* ============================================= Top-15 + sentinel variant"

MUTANTS = {
    "exponent shift": ("return (uint8_t)((x >> 2) & 0x1F);", "return (uint8_t)((x >> 3) & 0x1F);"),
    "sign bit of the field": ("(uint8_t)(((x >> 5) & 4) | (x & 3))", "(uint8_t)(((x >> 6) & 4) | (x & 3))"),
    "mantissa mask in rebuild": ("((e & 0x1F) << 2) | (a & 3));", "((e & 0x1F) << 2) | (a & 1));"),
    "field order in a group": ("word |= (uint32_t)e5m2_sign_mantissa(x[i]) << bit;",
                               "word |= (uint32_t)e5m2_sign_mantissa(x[i]) << (21 - bit);"),
    "group stride": ("uint8_t *w = A + 3 * (i / 8);\n        uint32_t word = (uint32_t)w[0] | ((uint32_t)w[1] << 8) | ((uint32_t)w[2] << 16);\n        word |=",
                     "uint8_t *w = A + 3 * (i / 16);\n        uint32_t word = (uint32_t)w[0] | ((uint32_t)w[1] << 8) | ((uint32_t)w[2] << 16);\n        word |="),
    "histogram bin": ("hist[e5m2_exponent(x[i])]++;", "hist[e5m2_exponent(x[i]) & 0xF]++;"),
    "field section size": ("L.off_b = L.off_a + pad16(3 * ((n + 7) / 8));", "L.off_b = L.off_a + pad16(n);"),
    "escape fix-up keeps the old exponent": ("x[start + pos] = (uint8_t)((x[start + pos] & 0x83) | ((block[2 * k + j] & 0x1F) << 2));",
                                             "x[start + pos] = (uint8_t)(x[start + pos] | ((block[2 * k + j] & 0x1F) << 2));"),
    "magic": ('memcpy(out, "UZE1", 4);', 'memcpy(out, "UZP1", 4);'),
    "repeated positions accepted": ("if (j > 0 && pos <= get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;",
                                    "if (j > 0 && pos < get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;"),
    "offsets not checked": ("if (get_u32(C) != 0 || get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;",
                            "if (get_u32(C) > m) return ORC_ERR_CORRUPT;"),
}

BATTERY = r"""
import sys, importlib.util
sys.path.insert(0, {root!r}); sys.path.insert(0, {here!r})
import oracle
spec = importlib.util.spec_from_file_location("pins", {pins!r})
pins = importlib.util.module_from_spec(spec); spec.loader.exec_module(pins)
o = oracle.Oracle(oracle.load({lib!r}))
checks = [
    lambda: pins.test_split_matches_binary16_semantics(o),
    lambda: pins.test_merge_inverts_split_and_is_a_bijection(o),
    lambda: pins.test_histogram_and_top16(o),
    lambda: pins.test_encode_matches_hand_worked_stream(o),
    lambda: pins.test_brute_force_tiny_streams(o, 24),
    lambda: pins.test_brute_force_tiny_streams(o, 1024),
    lambda: pins.test_closed_forms(o),
    lambda: pins.test_corrupt_streams_are_refused(o),
]
failed = []
for i, c in enumerate(checks):
    try:
        c()
    except Exception as ex:
        failed.append((i, type(ex).__name__))
print("FAILED", failed)
sys.exit(1 if failed else 0)
"""


def _run_battery(lib_path):
    code = BATTERY.format(root=os.path.dirname(HERE), here=HERE, lib=lib_path,
                          pins=os.path.join(HERE, "test_oracle_e5m2_pins.py"))
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)


def test_battery_passes_on_the_real_oracle():
    r = _run_battery(oracle.build())
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "uzip_oracle.c")).read()
    head, tail = src.split(E5M2_MARKER, 1)
    part, rest = tail.split(SENTINEL_MARKER, 1)  # the E5M2 part only
    assert part.count(old) == 1, f"mutation site for {name!r} not unique"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(head + E5M2_MARKER + part.replace(old, new) + SENTINEL_MARKER + rest)
    lib = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / "libmutant.so"))
    r = _run_battery(lib)
    assert r.returncode != 0, f"mutant {name!r} survived the pins:\n{r.stdout}{r.stderr}"
