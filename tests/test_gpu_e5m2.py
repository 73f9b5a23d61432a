"""GPU parity of the FP8 E5M2 codec (SplitZip review page, §4.2 / appendix C)
against the oracle's E5M2 variant, byte for byte: codebook tables, streams,
decoded values. Integer work: the tolerance is zero."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def check(uz, orc, x, exps, cb, chunk):
    xh = W.as_u8(x)
    rc, want = orc.e5m2_encode(xh, exps, chunk)
    assert rc == 0
    stream, nbytes = uz.e5m2_encode(x, cb, chunk)
    assert nbytes == want.size == uz.e5m2_compressed_size(xh.size, int.from_bytes(want[24:32].tobytes(), "little"),
                                                          chunk)
    got = stream[:nbytes].cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"stream differs at {bad.size} bytes, first at {bad[:8].tolist()} of {nbytes}")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = uz.e5m2_decode(stream, xh.size, stream_bytes=nbytes, status=status)
    assert int(status.item()) == 0 and np.array_equal(W.as_u8(y), xh)
    y2 = uz.e5m2_decode(torch.from_numpy(want).cuda(), xh.size, status=status)
    assert int(status.item()) == 0 and np.array_equal(W.as_u8(y2), xh)


def gpu_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def test_calibration_matches_oracle(uz, orc):
    x, s = W.workload_e5m2(device="cuda", small=True)
    cb = uz.e5m2_calibrate(s)
    exps = orc.e5m2_calibrate(W.as_u8(s))
    assert uz.codebook_exps(cb) == exps.tolist()
    assert uz.codebook_histogram(cb) == [int(v) for v in orc.e5m2_histogram(W.as_u8(s))]
    enc, dec, esc = orc.luts(exps)
    host = cb.cpu().numpy()
    assert np.array_equal(host[48:304], enc) and np.array_equal(host[32:48], dec)
    assert np.array_equal(host[304:560], esc)
    for n in (0, 1, 15, 16, 17, 1000, 65537):  # ragged sample tails
        xs = np.random.default_rng(n).integers(0, 256, n).astype(np.uint8)
        cbn = uz.e5m2_calibrate(gpu_u8(xs) if n else torch.empty(0, dtype=torch.uint8, device="cuda"))
        assert uz.codebook_exps(cbn) == orc.e5m2_calibrate(xs).tolist()


@pytest.mark.parametrize("chunk", [256, 1024, 4096])
def test_kv_small(uz, orc, chunk):
    x, s = W.workload_e5m2(device="cuda", small=True)
    cb = uz.e5m2_calibrate(s)
    check(uz, orc, x, orc.e5m2_calibrate(W.as_u8(s)), cb, chunk)


@pytest.mark.parametrize("chunk", [8, 24, 1000, 1024, 8200, 63496, 65536])
def test_edge_sizes(uz, orc, chunk):
    rng = np.random.default_rng(chunk)
    for n in sorted({1, 2, 7, 8, 9, 15, 31, 32, 33, chunk - 1, chunk, chunk + 1, 2047, 2048, 2049, 4095, 65537,
                     200_003}):
        if rng.random() < 0.5:
            xh = rng.integers(0, 256, n).astype(np.uint8)  # about half escapes
        else:
            xh = W.as_u8(W.to_e5m2_bits(torch.from_numpy(rng.standard_normal(n).astype(np.float32))))
        exps = rng.choice(32, 16, replace=False).astype(np.uint8)
        if rng.random() < 0.5:
            exps = orc.e5m2_calibrate(xh)
        check(uz, orc, gpu_u8(xh), exps, uz.codebook_from_exps(exps.tolist()), chunk)


def test_degenerate(uz, orc):
    n = 3 * 65536 + 11
    for xh in (np.zeros(n, np.uint8), np.full(n, 0x7C, np.uint8), np.tile(np.arange(256, dtype=np.uint8), n // 256 + 1)[:n]):
        for exps in (np.arange(16, dtype=np.uint8), orc.e5m2_calibrate(xh)):
            check(uz, orc, gpu_u8(xh), exps, uz.codebook_from_exps(exps.tolist()), 1024)
    x = torch.empty(0, dtype=torch.uint8, device="cuda")
    exps = np.arange(16, dtype=np.uint8)
    stream, nbytes = uz.e5m2_encode(x, uz.codebook_from_exps(exps.tolist()), 1024)
    assert np.array_equal(stream[:nbytes].cpu().numpy(), orc.e5m2_encode(np.zeros(0, np.uint8), exps, 1024)[1])


def test_streams_of_the_other_format_are_refused(uz):
    x = torch.randn(10_000, device="cuda").bfloat16()
    s16, n16 = uz.encode(x, uz.calibrate(x), 1024)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    uz.e5m2_decode(s16, 10_000, stream_bytes=n16, status=status)
    assert int(status.item()) == _lib.ERR_CORRUPT
    x8 = W.to_e5m2_bits(x)
    s8, n8 = uz.e5m2_encode(x8, uz.e5m2_calibrate(x8), 1024)
    uz.decode(s8, 10_000, stream_bytes=n8, status=status)
    assert int(status.item()) == _lib.ERR_CORRUPT


def test_kv_full(uz, orc):
    x, s = W.workload_e5m2(device="cuda")
    cb = uz.e5m2_calibrate(s)
    exps = orc.e5m2_calibrate(W.as_u8(s))
    check(uz, orc, x, exps, cb, 1024)
    del x
    torch.cuda.empty_cache()
