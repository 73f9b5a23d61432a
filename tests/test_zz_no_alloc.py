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
import os
import shutil
import subprocess

import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _encode_noalloc(lib, x, cb, chunk, sync=True):
    n = x.numel()
    cap = lib.uzip_compressed_size(n, n, chunk)
    out = torch.full((cap,), 0xAB, dtype=torch.uint8, device=x.device)
    nbytes = ctypes.c_size_t(0)
    rc = lib.uzip_encode_noalloc(_ptr(x) if n else None, n, chunk, _ptr(cb), _ptr(out), cap,
                                 ctypes.byref(nbytes) if sync else None, _stream())
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


def test_noalloc_asynchronous_calls_in_a_row(uz):
    """Without h_out_bytes the call does not wait: two calls with different
    inputs are enqueued back to back on one stream, the second reusing the
    scratch the first has just used, and the host synchronises once. Each
    stream (its size read from its own header) equals uzip_encode's."""
    lib = uz.load()
    x1 = W.heavy_tailed((1 << 21) + 3, seed=21, device="cuda")
    x2 = W.kv_cache((2, 2, 8, 512, 128), seed=22, device="cuda").reshape(-1)
    cb = uz.calibrate(W.gaussian(1 << 16, seed=23, device="cuda"))
    want1, n1 = uz.encode(x1, cb, 512)
    want2, n2 = uz.encode(x2, cb, 2048)
    rc1, got1, _ = _encode_noalloc(lib, x1, cb, 512, sync=False)
    rc2, got2, _ = _encode_noalloc(lib, x2, cb, 2048, sync=False)
    assert rc1 == _lib.OK and rc2 == _lib.OK
    torch.cuda.synchronize()
    for got, want, nb in ((got1, want1, n1), (got2, want2, n2)):
        assert uz.stream_info(got)["total_bytes"] == nb
        assert torch.equal(got[:nb], want[:nb])
        assert torch.all(got[nb:] == 0xAB)


def test_noalloc_empty_input(uz):
    """n = 0: a header and one zero offset, as uzip_encode writes them."""
    lib = uz.load()
    x = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    cb = uz.calibrate(W.gaussian(1 << 12, seed=24, device="cuda"))
    want, want_n = uz.encode(x, cb, 1024)
    rc, got, got_n = _encode_noalloc(lib, x, cb, 1024)
    assert rc == _lib.OK and got_n == want_n == lib.uzip_compressed_size(0, 0, 1024)
    assert torch.equal(got[:got_n], want[:want_n])


def test_noalloc_across_a_device_reset(tmp_path, uz):
    """A plain C program (tests/c/noalloc_reset.c, its own process) encodes
    with uzip_encode and uzip_encode_noalloc, calls cudaDeviceReset, and
    encodes again both ways: the no-alloc call must find its built-in scratch
    in the new context, and all four streams must be byte-identical."""
    from lossless_bf16_exponent_gb300 import build as B

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib = B.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "noalloc_reset")
    cuda = "/usr/local/cuda"
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(root, "tests", "c", "noalloc_reset.c"), "-o", exe,
           "-L", os.path.dirname(lib), "-luzip", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    for n, chunk in (("3000017", "1024"), ("65537", "256")):
        r = subprocess.run([exe, n, chunk], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stdout + r.stderr
        assert "noalloc_reset ok" in r.stdout
