"""CPU oracle for the fixed-length lossless BF16 exponent codec (SplitZip).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only code allowed to import
this package. The product (``lossless_bf16_exponent_gb300``) never imports it
and shares no code with it.

The arithmetic lives in ``uzip_oracle.c`` (plain scalar C, one loop per step of
the method as the SplitZip review page states it in §3.2-§3.4). This module
only compiles it with gcc and marshals numpy arrays through ctypes.

The FP8 E5M2 variant (the page's §4.2 / appendix C: the same Top-16
framework on E5M2 values) and the Top-15 + sentinel variant (§3.4, Table 6:
the alternative the page rejects) are in the same C file, after the BF16
codec.

Parity pins: every function is pinned against IEEE-754 semantics, the page's
closed-form sizes, hand-worked streams, exhaustive and brute-force checks --
the BF16 codec in ``tests/test_oracle_pins.py``, the E5M2 variant in
``tests/test_oracle_e5m2_pins.py``, the sentinel variant in
``tests/test_oracle_sentinel_pins.py`` (with planted-mistake batteries in the
matching ``*_mutants.py``); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "uzip_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, ERR_ARG, ERR_CHUNK, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 3, 4, 5

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle into a shared library (gcc, no CUDA)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src])
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and declare the C signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    u64, u32, p = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
    lib.orc_split.argtypes = [p, u64, p, p]
    lib.orc_merge.argtypes = [p, p, u64, p]
    lib.orc_histogram.argtypes = [p, u64, p]
    lib.orc_top16.argtypes = [p, p]
    lib.orc_luts.argtypes = [p, p, p, p]
    lib.orc_calibrate.argtypes = [p, u64, p]
    lib.orc_stream_bytes.argtypes = [u64, u64, u32]
    lib.orc_stream_bytes.restype = u64
    lib.orc_count_escapes.argtypes = [p, u64, p]
    lib.orc_count_escapes.restype = u64
    lib.orc_encode.argtypes = [p, u64, u32, p, p, u64, ctypes.POINTER(u64)]
    lib.orc_encode.restype = ctypes.c_int
    lib.orc_decode.argtypes = [p, u64, p, u64]
    lib.orc_decode.restype = ctypes.c_int
    lib.orc_e5m2_split.argtypes = [p, u64, p, p]
    lib.orc_e5m2_merge.argtypes = [p, p, u64, p]
    lib.orc_e5m2_histogram.argtypes = [p, u64, p]
    lib.orc_e5m2_calibrate.argtypes = [p, u64, p]
    lib.orc_e5m2_stream_bytes.argtypes = [u64, u64, u32]
    lib.orc_e5m2_stream_bytes.restype = u64
    lib.orc_e5m2_encode.argtypes = [p, u64, u32, p, p, u64, ctypes.POINTER(u64)]
    lib.orc_e5m2_encode.restype = ctypes.c_int
    lib.orc_e5m2_decode.argtypes = [p, u64, p, u64]
    lib.orc_e5m2_decode.restype = ctypes.c_int
    lib.orc_sentinel_luts.argtypes = [p, p, p, p]
    lib.orc_sentinel_stream_bytes.argtypes = [u64, u64, u32]
    lib.orc_sentinel_stream_bytes.restype = u64
    lib.orc_sentinel_encode.argtypes = [p, u64, u32, p, p, u64, ctypes.POINTER(u64)]
    lib.orc_sentinel_encode.restype = ctypes.c_int
    lib.orc_sentinel_decode.argtypes = [p, u64, p, u64]
    lib.orc_sentinel_decode.restype = ctypes.c_int
    for f in ("orc_split", "orc_merge", "orc_histogram", "orc_top16", "orc_luts", "orc_calibrate",
              "orc_e5m2_split", "orc_e5m2_merge", "orc_e5m2_histogram", "orc_e5m2_calibrate", "orc_sentinel_luts"):
        getattr(lib, f).restype = None
    if path is None:
        _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        x = x.view(np.uint16) if x.dtype.itemsize == 2 else x.astype(np.uint16)
    return x.reshape(-1)


class Oracle:
    """Thin numpy front end over one loaded copy of the C oracle."""

    def __init__(self, lib=None):
        self.lib = lib or load()

    def split(self, x):
        x = _u16(x)
        e = np.empty(x.size, np.uint8)
        a = np.empty(x.size, np.uint8)
        self.lib.orc_split(_ptr(x), x.size, _ptr(e), _ptr(a))
        return e, a

    def merge(self, a, e):
        a = np.ascontiguousarray(a, np.uint8)
        e = np.ascontiguousarray(e, np.uint8)
        x = np.empty(a.size, np.uint16)
        self.lib.orc_merge(_ptr(a), _ptr(e), a.size, _ptr(x))
        return x

    def histogram(self, x):
        x = _u16(x)
        h = np.zeros(256, np.uint64)
        self.lib.orc_histogram(_ptr(x), x.size, _ptr(h))
        return h

    def top16(self, hist):
        hist = np.ascontiguousarray(hist, np.uint64)
        exps = np.zeros(16, np.uint8)
        self.lib.orc_top16(_ptr(hist), _ptr(exps))
        return exps

    def luts(self, exps):
        exps = np.ascontiguousarray(exps, np.uint8)
        enc = np.zeros(256, np.uint8)
        dec = np.zeros(16, np.uint8)
        esc = np.zeros(256, np.uint8)
        self.lib.orc_luts(_ptr(exps), _ptr(enc), _ptr(dec), _ptr(esc))
        return enc, dec, esc

    def calibrate(self, sample):
        x = _u16(sample)
        exps = np.zeros(16, np.uint8)
        self.lib.orc_calibrate(_ptr(x), x.size, _ptr(exps))
        return exps

    def stream_bytes(self, n, m, chunk):
        return int(self.lib.orc_stream_bytes(n, m, chunk))

    def count_escapes(self, x, exps):
        x = _u16(x)
        exps = np.ascontiguousarray(exps, np.uint8)
        return int(self.lib.orc_count_escapes(_ptr(x), x.size, _ptr(exps)))

    def encode(self, x, exps, chunk=1024, cap=None):
        """Return (status, stream bytes as a uint8 array)."""
        x = _u16(x)
        exps = np.ascontiguousarray(exps, np.uint8)
        if cap is None:
            cap = self.stream_bytes(x.size, x.size, chunk) if 8 <= chunk <= 65536 and chunk % 8 == 0 else 64
        out = np.zeros(max(cap, 1), np.uint8)
        nbytes = ctypes.c_uint64(0)
        rc = self.lib.orc_encode(_ptr(x), x.size, chunk, _ptr(exps), _ptr(out), cap, ctypes.byref(nbytes))
        if rc != OK:
            return rc, None
        return rc, out[: nbytes.value].copy()

    def decode(self, stream, n):
        """Return (status, uint16 array of n values)."""
        s = np.ascontiguousarray(stream, np.uint8)
        x = np.zeros(max(n, 1), np.uint16)
        rc = self.lib.orc_decode(_ptr(s), s.size, _ptr(x), n)
        return rc, x[:n]

    # ------------------------------------------------ FP8 E5M2 (page §4.2, appendix C)

    def e5m2_split(self, x):
        x = np.ascontiguousarray(x, np.uint8).reshape(-1)
        e = np.empty(x.size, np.uint8)
        a = np.empty(x.size, np.uint8)
        self.lib.orc_e5m2_split(_ptr(x), x.size, _ptr(e), _ptr(a))
        return e, a

    def e5m2_merge(self, a, e):
        a = np.ascontiguousarray(a, np.uint8)
        e = np.ascontiguousarray(e, np.uint8)
        x = np.empty(a.size, np.uint8)
        self.lib.orc_e5m2_merge(_ptr(a), _ptr(e), a.size, _ptr(x))
        return x

    def e5m2_histogram(self, x):
        x = np.ascontiguousarray(x, np.uint8).reshape(-1)
        h = np.zeros(256, np.uint64)
        self.lib.orc_e5m2_histogram(_ptr(x), x.size, _ptr(h))
        return h

    def e5m2_calibrate(self, sample):
        x = np.ascontiguousarray(sample, np.uint8).reshape(-1)
        exps = np.zeros(16, np.uint8)
        self.lib.orc_e5m2_calibrate(_ptr(x), x.size, _ptr(exps))
        return exps

    def e5m2_stream_bytes(self, n, m, chunk):
        return int(self.lib.orc_e5m2_stream_bytes(n, m, chunk))

    def e5m2_encode(self, x, exps, chunk=1024, cap=None):
        """Return (status, stream bytes as a uint8 array)."""
        x = np.ascontiguousarray(x, np.uint8).reshape(-1)
        exps = np.ascontiguousarray(exps, np.uint8)
        if cap is None:
            cap = self.e5m2_stream_bytes(x.size, x.size, chunk) if 8 <= chunk <= 65536 and chunk % 8 == 0 else 64
        out = np.zeros(max(cap, 1), np.uint8)
        nbytes = ctypes.c_uint64(0)
        rc = self.lib.orc_e5m2_encode(_ptr(x), x.size, chunk, _ptr(exps), _ptr(out), cap, ctypes.byref(nbytes))
        if rc != OK:
            return rc, None
        return rc, out[: nbytes.value].copy()

    def e5m2_decode(self, stream, n):
        """Return (status, uint8 array of n E5M2 values)."""
        s = np.ascontiguousarray(stream, np.uint8)
        x = np.zeros(max(n, 1), np.uint8)
        rc = self.lib.orc_e5m2_decode(_ptr(s), s.size, _ptr(x), n)
        return rc, x[:n]

    # ------------------------------------------- Top-15 + sentinel (page §3.4, Table 6)

    def sentinel_luts(self, exps):
        exps = np.ascontiguousarray(exps, np.uint8)
        enc = np.zeros(256, np.uint8)
        dec = np.zeros(16, np.uint8)
        esc = np.zeros(256, np.uint8)
        self.lib.orc_sentinel_luts(_ptr(exps), _ptr(enc), _ptr(dec), _ptr(esc))
        return enc, dec, esc

    def sentinel_stream_bytes(self, n, m, chunk):
        return int(self.lib.orc_sentinel_stream_bytes(n, m, chunk))

    def sentinel_encode(self, x, exps, chunk=1024, cap=None):
        """Return (status, stream bytes); exps: the codebook's first 15 are used."""
        x = _u16(x)
        exps = np.ascontiguousarray(exps, np.uint8)
        if cap is None:
            cap = self.sentinel_stream_bytes(x.size, x.size, chunk) if 8 <= chunk <= 65536 and chunk % 8 == 0 else 64
        out = np.zeros(max(cap, 1), np.uint8)
        nbytes = ctypes.c_uint64(0)
        rc = self.lib.orc_sentinel_encode(_ptr(x), x.size, chunk, _ptr(exps), _ptr(out), cap, ctypes.byref(nbytes))
        if rc != OK:
            return rc, None
        return rc, out[: nbytes.value].copy()

    def sentinel_decode(self, stream, n):
        s = np.ascontiguousarray(stream, np.uint8)
        x = np.zeros(max(n, 1), np.uint16)
        rc = self.lib.orc_sentinel_decode(_ptr(s), s.size, _ptr(x), n)
        return rc, x[:n]
