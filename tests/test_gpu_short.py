"""Short inputs (at most 32 units of 2048 values and 4096 chunks) are encoded
by one CTA in one launch, with the escape lists in shared memory; mid-size
ones (at most 256 units and 4096 chunks) by one thread-block cluster of up to
16 CTAs, which exchange their escape counts through distributed shared
memory; longer ones by the dense and escape kernels. All must give the
oracle's stream byte for byte (SplitZip review page, §3.2), in all three
formats, on both sides of every limit, with chunks that span several of a
cluster's CTAs, with units whose escapes overflow their list, and with an
output buffer too small for the escapes. Integer work: the tolerance is
zero."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def _gauss(rng, n):
    return (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16(xh):
    return torch.from_numpy(np.ascontiguousarray(xh).view(np.int16)).cuda().view(torch.bfloat16)


def _check(uz, orc, xh, exps, chunk, fmt):
    n = xh.size
    if fmt == "e5m2":
        rc, want = orc.e5m2_encode(xh, exps, chunk)
        cb = uz.codebook_from_exps([int(v) for v in exps])
        x = torch.from_numpy(xh).cuda()
        stream, nbytes = uz.e5m2_encode(x, cb, chunk)
        dec = lambda s, nb: W.as_u8(uz.e5m2_decode(s, n, stream_bytes=nb, status=status))
    elif fmt == "sentinel":
        rc, want = orc.sentinel_encode(xh, exps, chunk)
        cb = uz.make_sentinel(uz.codebook_from_exps([int(v) for v in exps]))
        x = _bf16(xh)
        stream, nbytes = uz.sentinel_encode(x, cb, chunk)
        dec = lambda s, nb: W.as_u16(uz.sentinel_decode(s, n, stream_bytes=nb, status=status))
    else:
        rc, want = orc.encode(xh, exps, chunk)
        cb = uz.codebook_from_exps([int(v) for v in exps])
        x = _bf16(xh)
        stream, nbytes = uz.encode(x, cb, chunk)
        dec = lambda s, nb: W.as_u16(uz.decode(s, n, stream_bytes=nb, status=status))
    assert rc == 0
    assert nbytes == want.size
    got = stream[:nbytes].cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"{fmt} n={n} chunk={chunk}: stream differs at {bad.size} bytes, first {bad[:8].tolist()}")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert np.array_equal(dec(stream, nbytes), xh) and int(status.item()) == 0


@pytest.mark.parametrize("fmt", ["bf16", "e5m2", "sentinel"])
@pytest.mark.parametrize("chunk,sizes", [
    (1024, [2047, 2048, 2049, 65535, 65536, 65537, 67584]),  # 32 units: the last short input is 65,536 values
    (8, [32767, 32768, 32769, 32776]),                        # 4096 chunks: the last short input is 32,768
    (24, [24 * 4096, 24 * 4096 + 1]),
    (65536, [1, 65536, 65537]),
])
def test_both_sides_of_the_boundary(uz, orc, fmt, chunk, sizes):
    rng = np.random.default_rng(chunk)
    for n in sizes:
        if fmt == "e5m2":
            xh = rng.integers(0, 256, n).astype(np.uint8)
            xh[rng.random(n) < 0.7] = 0x3C  # skewed, so a codebook leaves some escapes
            exps = orc.e5m2_calibrate(xh[: max(1, n // 2)])
        else:
            xh = _gauss(rng, n)
            xh[rng.integers(0, n, max(1, n // 40))] = 0x7F80  # Inf: escapes
            exps = orc.calibrate(_gauss(rng, 1 << 14))
        _check(uz, orc, xh, exps, chunk, fmt)


@pytest.mark.parametrize("fmt", ["bf16", "e5m2", "sentinel"])
@pytest.mark.parametrize("chunk,sizes", [
    (1024, [33 * 2048 - 5, 48 * 2048, 96 * 2048 + 7, 256 * 2048, 256 * 2048 + 1]),  # 256 units: the last cluster input
    (104, [409600]),                 # 3939 chunks: a cluster
    (96, [409600]),                  # 4267 chunks: the two kernels
    (128, [4096 * 128, 4096 * 128 + 8]),
    (65536, [40 * 2048, 100 * 2048 + 3]),  # one chunk over many CTAs of the cluster
    (8200, [77 * 2048 + 11]),        # chunks crossing the CTAs' boundaries
])
def test_both_sides_of_the_cluster_limits(uz, orc, fmt, chunk, sizes):
    rng = np.random.default_rng(chunk + 5)
    for n in sizes:
        if fmt == "e5m2":
            xh = rng.integers(0, 256, n).astype(np.uint8)
            xh[rng.random(n) < 0.7] = 0x3C
            exps = orc.e5m2_calibrate(xh[: max(1, n // 2)])
        else:
            xh = _gauss(rng, n)
            xh[rng.integers(0, n, max(1, n // 40))] = 0x7F80
            exps = orc.calibrate(_gauss(rng, 1 << 14))
        _check(uz, orc, xh, exps, chunk, fmt)


@pytest.mark.parametrize("fmt", ["bf16", "e5m2", "sentinel"])
@pytest.mark.parametrize("chunk", [8, 1000, 2048])
def test_units_whose_escapes_overflow_their_list(uz, orc, fmt, chunk):
    """Every unit, or every other one, holds more escapes than its list (64):
    the one-CTA and cluster encoders place them from their mask bits and the
    input (chunk 8 on the longer input: more than 4096 chunks, the two
    kernels)."""
    rng = np.random.default_rng(chunk + 3)
    for n in (20 * 2048 + 333, 100 * 2048 + 333):  # one CTA; a cluster of 15
        _overflowing(uz, orc, fmt, chunk, rng, n)


def _overflowing(uz, orc, fmt, chunk, rng, n):
    if fmt == "e5m2":
        xh = rng.integers(0, 256, n).astype(np.uint8)
        exps = np.arange(16, dtype=np.uint8)
        xh[: n // 2 : 2] = 0x3C  # exponent 15: coded; the rest mostly escapes
    else:
        xh = rng.integers(0, 65536, n).astype(np.uint16)  # random patterns: ~94 % escapes
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        xh[2048:4096] = 0x3F80  # one unit without escapes if 0x7F is not coded
    _check(uz, orc, xh, exps, chunk, fmt)


@pytest.mark.parametrize("n", [40_000, 300_000])  # one CTA; a cluster
def test_capacity_overflow_of_a_short_input(uz, n):
    x = W.heavy_tailed(n, seed=8, device="cuda")
    cb = uz.calibrate(W.gaussian(1 << 16, seed=9, device="cuda"))
    n = x.numel()
    cap = uz.compressed_size(n, 0, 1024) + 30  # room for 10 escapes only
    out = torch.full((cap + 4096,), 0xAB, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.UzipError) as e:
        uz.encode(x, cb, 1024, out=out[:cap])
    assert e.value.code == _lib.ERR_CAPACITY
    assert torch.all(out[cap:] == 0xAB)
    assert uz.stream_info(out, cap)["flags"] & _lib.FLAG_CAPACITY
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    uz.decode(out, n, status=status, stream_bytes=cap)
    assert int(status.item()) == _lib.ERR_CORRUPT
