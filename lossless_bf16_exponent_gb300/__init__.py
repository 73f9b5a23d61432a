"""uzip: fixed-length lossless BF16 exponent codec (SplitZip) for NVIDIA GB300.

The codec itself is ``libuzip.so`` (hand-written CUDA for sm_103a, C ABI in
``include/uzip.h``); this package holds its build script, the ctypes / PyTorch
front end and the seeded synthetic workloads. Importing the package does not
load the library; the first codec call does, and fails loudly if it is
missing.
"""
from .codec import (CODEBOOK_BYTES, HEADER_BYTES, UzipError, calibrate, codebook_exps, codebook_from_exps,
                    codebook_histogram, compressed_size, decode, e5m2_calibrate, e5m2_compressed_size,
                    e5m2_decode, e5m2_encode, encode, encode_dynamic, load, make_sentinel, max_compressed_size,
                    new_codebook, roundtrip_ok, sentinel_compressed_size, sentinel_decode, sentinel_encode,
                    stream_copy, stream_info, workspace_bytes)

__all__ = [
    "CODEBOOK_BYTES", "HEADER_BYTES", "UzipError", "calibrate", "codebook_exps", "codebook_from_exps",
    "codebook_histogram", "compressed_size", "decode", "e5m2_calibrate", "e5m2_compressed_size", "e5m2_decode",
    "e5m2_encode", "encode", "encode_dynamic", "load", "make_sentinel", "max_compressed_size",
    "sentinel_compressed_size", "sentinel_decode", "sentinel_encode",
    "new_codebook", "roundtrip_ok", "stream_copy", "stream_info", "workspace_bytes",
]
