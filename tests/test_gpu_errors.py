"""Device-side error reporting, exercised without any GPU fault: every case
below keeps all reads and writes inside the buffers (the kernels bound-check
what a bad stream or a small buffer could push outside), no kernel waits on
another block, and the CUDA context stays usable afterwards."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def _data(n=1 << 20, seed=5):
    x = W.heavy_tailed(n, seed=seed, device="cuda")  # a few percent escapes
    cb_sample = W.gaussian(1 << 16, seed=7, device="cuda")
    return x, cb_sample


def test_nothing_written_past_the_stream(uz):
    x, s = _data()
    cb = uz.calibrate(s)
    out = torch.full((uz.max_compressed_size(x.numel(), 1024),), 0xAB, dtype=torch.uint8, device="cuda")
    _, nbytes = uz.encode(x, cb, 1024, out=out)
    assert torch.all(out[nbytes:] == 0xAB)


def test_capacity_overflow_is_flagged_and_bounded(uz):
    x, s = _data()
    cb = uz.calibrate(s)
    n = x.numel()
    cap = uz.compressed_size(n, 0, 1024) + 999  # room for 333 escapes only
    out = torch.full((cap + 4096,), 0xAB, dtype=torch.uint8, device="cuda")
    ws = torch.empty(uz.workspace_bytes(n, 1024), dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.UzipError) as e:
        uz.encode(x, cb, 1024, out=out[:cap], workspace=ws)
    assert e.value.code == _lib.ERR_CAPACITY
    assert torch.all(out[cap:] == 0xAB)  # nothing past the capacity
    info = uz.stream_info(out, cap)
    assert info["flags"] & _lib.FLAG_CAPACITY
    # a flagged stream is refused by the decoder
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full((n,), 7, dtype=torch.int16, device="cuda")
    uz.decode(out, n, out=y, status=status, stream_bytes=cap)
    assert int(status.item()) == _lib.ERR_CORRUPT
    assert torch.all(y == 7)


def test_context_survives_a_flagged_encode(uz):
    """After a device-side error the CUDA context stays usable."""
    x, s = _data()
    cb = uz.calibrate(s)
    n = x.numel()
    cap = uz.compressed_size(n, 0, 1024)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.UzipError):
        uz.encode(x, cb, 1024, out=out)
    torch.cuda.synchronize()
    assert uz.roundtrip_ok(x, cb, 1024)


def _good_stream(uz, n=200_000):
    x, s = _data(n)
    cb = uz.calibrate(s)
    stream, nbytes = uz.encode(x, cb, 1024)
    return x, stream[:nbytes].clone(), nbytes


def _decode_status(uz, stream, n, nbytes=None):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = torch.full((max(n, 1),), 7, dtype=torch.int16, device="cuda")[:n]
    uz.decode(stream, n, out=y, status=status, stream_bytes=nbytes)
    return int(status.item()), y


@pytest.mark.parametrize("what", ["magic", "version", "flags", "n", "chunk", "nc", "m", "total"])
def test_corrupt_header_writes_nothing(uz, what):
    x, s, nb = _good_stream(uz)
    field = {"magic": 0, "version": 4, "flags": 6, "n": 8, "chunk": 16, "nc": 20, "m": 24, "total": 48}[what]
    s[field] ^= 0x5
    st, y = _decode_status(uz, s, x.numel())
    assert st == _lib.ERR_CORRUPT
    assert torch.all(y == 7)


def test_wrong_n_and_short_stream(uz):
    x, s, nb = _good_stream(uz)
    assert _decode_status(uz, s, x.numel() - 1)[0] == _lib.ERR_CORRUPT
    st, y = _decode_status(uz, s, x.numel(), nbytes=nb - 1)
    assert st == _lib.ERR_CORRUPT and torch.all(y == 7)
    assert _decode_status(uz, s, x.numel())[0] == _lib.OK


def _sections(n, chunk=1024):
    pad = lambda v: (v + 15) // 16 * 16
    nc = -(-n // chunk)
    off_c = 64 + pad(n) + pad((n + 1) // 2)
    return off_c, off_c + pad(4 * (nc + 1)), nc


def test_bad_escape_position_is_reported(uz):
    x, s, nb = _good_stream(uz)
    off_c, off_d, nc = _sections(x.numel())
    offs = s[off_c:off_c + 4 * (nc + 1)].cpu().numpy().view("<u4")
    c = int(np.flatnonzero(np.diff(offs) > 0)[0])  # a chunk with escapes
    p = off_d + 3 * int(offs[c])
    s[p], s[p + 1] = 0xFF, 0xFF  # position 65535 >= chunk
    assert _decode_status(uz, s, x.numel())[0] == _lib.ERR_CORRUPT


def test_offsets_not_rising_are_reported(uz):
    x, s, nb = _good_stream(uz)
    off_c, off_d, nc = _sections(x.numel())
    s[off_c + 4 * 5:off_c + 4 * 6] = torch.tensor([0xFF, 0xFF, 0xFF, 0x7F], dtype=torch.uint8, device="cuda")
    assert _decode_status(uz, s, x.numel())[0] == _lib.ERR_CORRUPT
