"""uzip_encode_noalloc: the encoder for callers that cannot allocate device
memory for a workspace (its workspace is an array built into the library).

This file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test. Each call goes
through the C ABI and must produce exactly the bytes uzip_encode produces for
the same input -- the codec is lossless integer work, so the tolerance is
zero -- over several calls in a row, since every call reuses the same
built-in scratch array.
"""
import ctypes

import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _encode_noalloc(lib, x, cb, chunk):
    n = x.numel()
    cap = lib.uzip_compressed_size(n, n, chunk)
    out = torch.full((cap,), 0xAB, dtype=torch.uint8, device=x.device)
    nbytes = ctypes.c_size_t(0)
    rc = lib.uzip_encode_noalloc(_ptr(x), n, chunk, _ptr(cb), _ptr(out), cap, ctypes.byref(nbytes), _stream())
    return rc, out, nbytes.value


def test_noalloc_matches_uzip_encode_on_consecutive_calls(uz):
    lib = uz.load()
    cases = [
        # a KV-shaped tensor of 12.6 M values (few escapes) ...
        (W.kv_cache((8, 2, 8, 768, 128), seed=11, device="cuda").reshape(-1), W.kv_cache_sample(device="cuda"), 1024),
        # ... then a smaller, escape-heavy one with another chunk size: the
        # scratch still holds the first call's data
        (W.heavy_tailed((1 << 20) + 37, seed=12, device="cuda"), W.gaussian(1 << 16, seed=13, device="cuda"), 256),
        # ... then the first one again
        None,
    ]
    cases[2] = cases[0]
    for x, sample, chunk in cases:
        cb = uz.calibrate(sample)
        want, want_n = uz.encode(x, cb, chunk)
        rc, got, got_n = _encode_noalloc(lib, x, cb, chunk)
        assert rc == _lib.OK
        assert got_n == want_n
        assert torch.equal(got[:got_n], want[:want_n])
        assert torch.all(got[got_n:] == 0xAB)  # nothing written past the stream
        y = uz.decode(got, x.numel(), stream_bytes=got_n)
        assert torch.equal(y.view(torch.int16), x.view(torch.int16))


def test_noalloc_at_its_maximum_size(uz):
    lib = uz.load()
    x = W.gaussian(_lib.NOALLOC_MAX_N, seed=14, device="cuda")
    cb = uz.calibrate(W.gaussian(1 << 16, seed=15, device="cuda"))
    want, want_n = uz.encode(x, cb, 4096)
    rc, got, got_n = _encode_noalloc(lib, x, cb, 4096)
    assert rc == _lib.OK and got_n == want_n
    assert torch.equal(got[:got_n], want[:want_n])
    del x, want, got
    torch.cuda.empty_cache()


def test_noalloc_rejects_sizes_beyond_its_scratch(uz):
    lib = uz.load()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    rc = lib.uzip_encode_noalloc(fake, _lib.NOALLOC_MAX_N + 1, 1024, fake, fake, 1 << 40, None, None)
    assert rc == _lib.ERR_CAPACITY
