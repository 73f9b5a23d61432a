"""bench.py reports a kernel's DRAM traffic from a committed ncu summary only
while the kernel code that summary was taken on is unchanged: the check
hashes the kernel's CUDA source and the headers it includes, with comments
and whitespace removed."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _hash_of(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return bench.source_code_hash(str(p))


def test_code_hash_ignores_comments_and_layout(tmp_path):
    a = _hash_of(tmp_path, "a.cu", "int f(int x) {\n    return x + 1;  // one more\n}\n")
    b = _hash_of(tmp_path, "b.cu", "/* a note\n   over lines */\nint f(int x)\n{ return x + 1; }\n")
    assert a == b


def test_code_hash_sees_code_changes(tmp_path):
    a = _hash_of(tmp_path, "a.cu", "int f(int x) { return x + 1; }\n")
    b = _hash_of(tmp_path, "b.cu", "int f(int x) { return x + 2; }\n")
    assert a != b


def test_traffic_needs_a_matching_summary(tmp_path, monkeypatch):
    # A summary whose code hash does not match the source gives no traffic.
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "encode_kv_cache.md").write_text("dram_bytes_per_full_launch: 123\ncode_sha256_16: 0000000000000000\n")
    csrc = tmp_path / "lossless_bf16_exponent_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (csrc / "encode.cu").write_text("int f() { return 0; }\n")
    (csrc / "uzip_internal.cuh").write_text("#pragma once\n")
    (tmp_path / "include" / "uzip.h").write_text("#define UZIP_VERSION 1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("encode") is None
    good = bench.kernel_code_hash("encode.cu")
    (prof / "encode_kv_cache.md").write_text(f"dram_bytes_per_full_launch: 123\ncode_sha256_16: {good}\n")
    assert bench.profile_traffic("encode") == 123
    # a change in an included header is a change of the kernel code
    (csrc / "uzip_internal.cuh").write_text("#pragma once\nconstexpr int k = 1;\n")
    assert bench.profile_traffic("encode") is None
