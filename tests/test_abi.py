"""C-ABI checks that need no GPU: libuzip.so builds for sm_103a, loads, exports
every entry point include/uzip.h declares, and its host-only paths (exact
sizes, argument validation) behave as documented. No kernel is launched."""
import ctypes
import os
import re

import pytest

from lossless_bf16_exponent_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "uzip.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"UZIP_API\s+[\w\s\*]+?\b(uzip_\w+)\s*\(", text)))


def test_header_declares_the_documented_api():
    syms = declared_symbols()
    for name in ("uzip_calibrate", "uzip_encode", "uzip_decode", "uzip_compressed_size"):
        assert name in syms
    assert set(syms) == set(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and nothing else leaks from the library's C++ internals
    nm = os.popen(f"nm -D --defined-only {_lib.lib_path()}").read()
    exported = {l.split()[-1] for l in nm.splitlines() if " T " in l}
    assert {s for s in exported if s.startswith("uzip_")} == set(declared_symbols())


def test_built_for_sm_103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version_and_status_strings(lib):
    assert lib.uzip_version() == 1
    for code in range(8):
        assert lib.uzip_status_string(code)
    assert lib.uzip_status_string(0) == b"ok"


def pad16(v):
    return (v + 15) // 16 * 16


@pytest.mark.parametrize("chunk", [8, 24, 256, 1024, 4096, 65536])
def test_compressed_size_matches_format_and_oracle(lib, orc, chunk):
    for n in (0, 1, 2, 7, 8, 9, chunk - 1, chunk, chunk + 1, 10 ** 6 + 3, (1 << 28), 0xFFFFFFFF):
        nc = -(-n // chunk)
        for m in {0, 1, n // 3, n}:
            if m > n:
                continue
            want = 64 + pad16(n) + pad16((n + 1) // 2) + pad16(4 * (nc + 1)) + 3 * m
            assert lib.uzip_compressed_size(n, m, chunk) == want
            assert orc.stream_bytes(n, m, chunk) == want


def test_compressed_size_rejects_invalid(lib):
    assert lib.uzip_compressed_size(100, 0, 0) == 0
    assert lib.uzip_compressed_size(100, 0, 12) == 0
    assert lib.uzip_compressed_size(100, 0, 65544) == 0
    assert lib.uzip_compressed_size(100, 101, 1024) == 0
    assert lib.uzip_compressed_size(1 << 32, 0, 1024) == 0
    assert lib.uzip_encode_workspace_bytes(100, 12) == 0
    assert lib.uzip_encode_workspace_bytes(1 << 32, 1024) == 0
    units = -(-(1 << 28) // 1024) // 1024  # at least one descriptor per 1024 chunks
    assert lib.uzip_encode_workspace_bytes(1 << 28, 1024) >= 64 + 8 * units


# Host-side validation returns before any CUDA call, so fake pointers are
# never dereferenced.
A16, MIS = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)


def test_encode_argument_validation(lib):
    sz = ctypes.c_size_t
    ws = lib.uzip_encode_workspace_bytes(1000, 1024)
    cap = lib.uzip_compressed_size(1000, 1000, 1024)
    enc = lambda *a: lib.uzip_encode(*a, None, None)
    assert enc(A16, 1000, 12, A16, A16, cap, A16, ws) == _lib.ERR_CHUNK
    assert enc(A16, 1000, 0, A16, A16, cap, A16, ws) == _lib.ERR_CHUNK
    assert enc(None, 1000, 1024, A16, A16, cap, A16, ws) == _lib.ERR_ARG
    assert enc(A16, 1000, 1024, None, A16, cap, A16, ws) == _lib.ERR_ARG
    assert enc(A16, 1000, 1024, A16, None, cap, A16, ws) == _lib.ERR_ARG
    assert enc(A16, 1000, 1024, A16, A16, cap, None, ws) == _lib.ERR_ARG
    assert enc(A16, 1 << 32, 1024, A16, A16, cap, A16, ws) == _lib.ERR_ARG
    assert enc(MIS, 1000, 1024, A16, A16, cap, A16, ws) == _lib.ERR_ALIGN
    assert enc(A16, 1000, 1024, MIS, A16, cap, A16, ws) == _lib.ERR_ALIGN
    assert enc(A16, 1000, 1024, A16, MIS, cap, A16, ws) == _lib.ERR_ALIGN
    assert enc(A16, 1000, 1024, A16, A16, cap, MIS, ws) == _lib.ERR_ALIGN
    fixed = lib.uzip_compressed_size(1000, 0, 1024)
    assert enc(A16, 1000, 1024, A16, A16, fixed - 1, A16, ws) == _lib.ERR_CAPACITY
    assert enc(A16, 1000, 1024, A16, A16, cap, A16, ws - 1) == _lib.ERR_CAPACITY


def test_noalloc_encode_rejects_oversize_before_any_cuda_call(lib):
    n = _lib.NOALLOC_MAX_N
    assert lib.uzip_encode_noalloc(A16, n + 1, 1024, A16, A16, 1 << 40, None, None) == _lib.ERR_CAPACITY
    assert lib.uzip_encode_noalloc(A16, n, 12, A16, A16, 1 << 40, None, None) == _lib.ERR_CHUNK


def test_decode_and_info_argument_validation(lib):
    assert lib.uzip_decode(None, 1000, A16, 10, None, None) == _lib.ERR_ARG
    assert lib.uzip_decode(A16, 1000, None, 10, None, None) == _lib.ERR_ARG
    assert lib.uzip_decode(A16, 1000, A16, 1 << 32, None, None) == _lib.ERR_ARG
    assert lib.uzip_decode(MIS, 1000, A16, 10, None, None) == _lib.ERR_ALIGN
    assert lib.uzip_decode(A16, 1000, MIS, 10, None, None) == _lib.ERR_ALIGN
    assert lib.uzip_decode(A16, 1000, A16, 10, ctypes.c_void_p(0x10002), None) == _lib.ERR_ALIGN
    assert lib.uzip_decode(A16, 63, A16, 10, None, None) == _lib.ERR_CAPACITY
    info = _lib.Info()
    assert lib.uzip_stream_info(None, 100, ctypes.byref(info), None) == _lib.ERR_ARG
    assert lib.uzip_stream_info(MIS, 100, ctypes.byref(info), None) == _lib.ERR_ALIGN
    assert lib.uzip_stream_info(A16, 63, ctypes.byref(info), None) == _lib.ERR_CORRUPT


def test_calibrate_and_codebook_validation(lib):
    assert lib.uzip_calibrate(A16, 100, None, None) == _lib.ERR_ARG
    assert lib.uzip_calibrate(None, 100, A16, None) == _lib.ERR_ARG
    assert lib.uzip_calibrate(MIS, 100, A16, None) == _lib.ERR_ALIGN
    assert lib.uzip_calibrate(A16, 100, MIS, None) == _lib.ERR_ALIGN
    dup = (ctypes.c_uint8 * 16)(*([1] * 16))
    assert lib.uzip_codebook_from_exps(dup, A16, None) == _lib.ERR_ARG
    ok = (ctypes.c_uint8 * 16)(*range(16))
    assert lib.uzip_codebook_from_exps(ok, MIS, None) == _lib.ERR_ALIGN
    assert lib.uzip_codebook_from_exps(None, A16, None) == _lib.ERR_ARG


def test_stream_copy_argument_validation(lib):
    # Checked on the host before the memory kinds are looked up or anything is launched.
    assert lib.uzip_stream_copy(None, A16, 4096, None, None) == _lib.ERR_ARG
    assert lib.uzip_stream_copy(A16, None, 4096, None, None) == _lib.ERR_ARG
    assert lib.uzip_stream_copy(MIS, A16, 4096, None, None) == _lib.ERR_ALIGN
    assert lib.uzip_stream_copy(A16, MIS, 4096, None, None) == _lib.ERR_ALIGN
    assert lib.uzip_stream_copy(A16, A16, 4096, ctypes.c_void_p(0x10004), None) == _lib.ERR_ALIGN
    assert lib.uzip_stream_copy(A16, A16, 63, None, None) == _lib.ERR_CAPACITY
