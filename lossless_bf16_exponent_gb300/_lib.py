"""ctypes declarations of libuzip's C ABI (``include/uzip.h``).

Argument marshalling only: every step of the codec runs in the library's CUDA
kernels. A missing library is an error, never a silent fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

OK, ERR_ARG, ERR_ALIGN, ERR_CHUNK, ERR_CAPACITY, ERR_CORRUPT, ERR_TIMEOUT, ERR_CUDA = range(8)
HEADER_BYTES = 64
CODEBOOK_BYTES = 4096
CB_EXPS, CB_DEC, CB_ENC, CB_ESC, CB_HIST = 16, 32, 48, 304, 1024
FLAG_CAPACITY = 0x1
FORMAT_BF16, FORMAT_E5M2, FORMAT_SENTINEL = range(3)
MAX_N = 0xFFFFFFFF

EXPORTS = (
    "uzip_calibrate", "uzip_codebook_from_exps", "uzip_compressed_size", "uzip_encode_workspace_bytes",
    "uzip_encode", "uzip_encode_noalloc", "uzip_encode_dynamic", "uzip_decode", "uzip_stream_copy",
    "uzip_stream_info", "uzip_status_string", "uzip_e5m2_calibrate", "uzip_e5m2_compressed_size",
    "uzip_e5m2_encode", "uzip_e5m2_decode", "uzip_codebook_make_sentinel", "uzip_sentinel_compressed_size",
    "uzip_sentinel_encode", "uzip_sentinel_decode",
    "uzip_version",
)
NOALLOC_MAX_N = 1 << 25


class Info(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_uint64), ("escapes", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64),
        ("payload_bytes", ctypes.c_uint64), ("chunk", ctypes.c_uint32), ("nc", ctypes.c_uint32),
        ("version", ctypes.c_uint32), ("flags", ctypes.c_uint32), ("exps", ctypes.c_uint8 * 16),
        ("format", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
    ]


class UzipError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libuzip.so (in-tree). Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libuzip.so not found at {p}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(p)
    vp, sz, u32, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_int
    L.uzip_calibrate.argtypes = [vp, sz, vp, vp]
    L.uzip_codebook_from_exps.argtypes = [ctypes.POINTER(ctypes.c_uint8), vp, vp]
    L.uzip_compressed_size.argtypes = [sz, sz, u32]
    L.uzip_compressed_size.restype = sz
    L.uzip_encode_workspace_bytes.argtypes = [sz, u32]
    L.uzip_encode_workspace_bytes.restype = sz
    L.uzip_encode.argtypes = [vp, sz, u32, vp, vp, sz, vp, sz, ctypes.POINTER(sz), vp]
    L.uzip_encode_noalloc.argtypes = [vp, sz, u32, vp, vp, sz, ctypes.POINTER(sz), vp]
    L.uzip_encode_dynamic.argtypes = [vp, sz, u32, vp, vp, sz, vp, sz, ctypes.POINTER(sz), vp]
    L.uzip_stream_copy.argtypes = [vp, vp, sz, vp, vp]
    L.uzip_e5m2_calibrate.argtypes = [vp, sz, vp, vp]
    L.uzip_e5m2_compressed_size.argtypes = [sz, sz, u32]
    L.uzip_e5m2_compressed_size.restype = sz
    L.uzip_e5m2_encode.argtypes = [vp, sz, u32, vp, vp, sz, vp, sz, ctypes.POINTER(sz), vp]
    L.uzip_e5m2_decode.argtypes = [vp, sz, vp, sz, vp, vp]
    L.uzip_codebook_make_sentinel.argtypes = [vp, vp]
    L.uzip_sentinel_compressed_size.argtypes = [sz, sz, u32]
    L.uzip_sentinel_compressed_size.restype = sz
    L.uzip_sentinel_encode.argtypes = [vp, sz, u32, vp, vp, sz, vp, sz, ctypes.POINTER(sz), vp]
    L.uzip_sentinel_decode.argtypes = [vp, sz, vp, sz, vp, vp]
    L.uzip_decode.argtypes = [vp, sz, vp, sz, vp, vp]
    L.uzip_stream_info.argtypes = [vp, sz, ctypes.POINTER(Info), vp]
    L.uzip_status_string.argtypes = [i]
    L.uzip_status_string.restype = ctypes.c_char_p
    L.uzip_version.argtypes = []
    for f in ("uzip_calibrate", "uzip_codebook_from_exps", "uzip_encode", "uzip_encode_noalloc",
              "uzip_encode_dynamic", "uzip_decode", "uzip_stream_copy", "uzip_stream_info", "uzip_version",
              "uzip_e5m2_calibrate", "uzip_e5m2_encode", "uzip_e5m2_decode", "uzip_codebook_make_sentinel",
              "uzip_sentinel_encode", "uzip_sentinel_decode"):
        getattr(L, f).restype = i
    if path is None:
        _lib = L
    return L


def status_string(code: int) -> str:
    try:
        return load().uzip_status_string(code).decode()
    except Exception:
        return "status"


def check(code: int, where: str) -> None:
    if code != OK:
        raise UzipError(code, where)
