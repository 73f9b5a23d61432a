"""The Top-15 + sentinel pins must catch plausible mistakes in the oracle's
sentinel variant: each case plants one mistake in a copy of the oracle's C
source (inside its sentinel part only), compiles it and runs the sentinel pin
battery in a child process; the case passes only if the battery fails."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SENTINEL_MARKER = "/* ============================================= Top-15 + sentinel variant"

MUTANTS = {
    "sentinel code not 15": ("        enc[v] = 15;\n        esc[v] = 1;", "        enc[v] = 14;\n        esc[v] = 1;"),
    "sixteen exponents coded": ("    for (int k = 0; k < 15; k++) {\n        enc[exps[k]]", "    for (int k = 0; k < 16; k++) {\n        enc[exps[k]]"),
    "value not the raw exponent": ("if (esc[e]) D[running++] = e;", "if (esc[e]) D[running++] = (uint8_t)(e ^ 1);"),
    "header keeps the 16th exponent": ("out[47] = 0;", "out[47] = exps[15];"),
    "decoder misses the sentinel": ("            if (code == 15) {", "            if (code == 14) {"),
    "nibble order": ("B[i / 2] = (uint8_t)(B[i / 2] | (code << (4 * (i % 2))));",
                     "B[i / 2] = (uint8_t)(B[i / 2] | (code << (4 * ((i + 1) % 2))));"),
    "three bytes per escape": ("return layout_of(n, chunk).off_d + m;", "return layout_of(n, chunk).off_d + 3 * m;"),
    "magic": ('memcpy(out, "UZS1", 4);', 'memcpy(out, "UZP1", 4);'),
}

BATTERY = r"""
import sys, importlib.util
sys.path.insert(0, {root!r}); sys.path.insert(0, {here!r})
import oracle
spec = importlib.util.spec_from_file_location("pins", {pins!r})
pins = importlib.util.module_from_spec(spec); spec.loader.exec_module(pins)
o = oracle.Oracle(oracle.load({lib!r}))
checks = [
    lambda: pins.test_encode_matches_hand_worked_stream(o),
    lambda: pins.test_luts(o),
    lambda: pins.test_brute_force_tiny_streams(o, 24),
    lambda: pins.test_brute_force_tiny_streams(o, 1024),
    lambda: pins.test_closed_forms_and_coverage(o),
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
                          pins=os.path.join(HERE, "test_oracle_sentinel_pins.py"))
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)


def test_battery_passes_on_the_real_oracle():
    r = _run_battery(oracle.build())
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "uzip_oracle.c")).read()
    head, tail = src.split(SENTINEL_MARKER, 1)
    assert tail.count(old) == 1, f"mutation site for {name!r} not unique"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(head + SENTINEL_MARKER + tail.replace(old, new))
    lib = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / "libmutant.so"))
    r = _run_battery(lib)
    assert r.returncode != 0, f"mutant {name!r} survived the pins:\n{r.stdout}{r.stderr}"
