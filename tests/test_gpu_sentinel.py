"""GPU parity of the Top-15 + sentinel codec (SplitZip review page, §3.4 and
Table 6: code 15 marks an escape and the decoder finds escapes by scanning the
code stream) against the oracle's sentinel variant, byte for byte: codebook
tables, streams, decoded values. Integer work: the tolerance is zero."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def bf16(xh):
    return torch.from_numpy(np.ascontiguousarray(xh, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def sentinel_codebook(uz, exps):
    return uz.make_sentinel(uz.codebook_from_exps([int(v) for v in exps]))


def check(uz, orc, x, exps, cb, chunk):
    xh = W.as_u16(x)
    n = xh.size
    rc, want = orc.sentinel_encode(xh, exps, chunk)
    assert rc == 0
    m = int.from_bytes(want[24:32].tobytes(), "little")
    stream, nbytes = uz.sentinel_encode(x, cb, chunk)
    assert nbytes == want.size == uz.sentinel_compressed_size(n, m, chunk)
    got = stream[:nbytes].cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"stream differs at {bad.size} bytes, first at {bad[:8].tolist()} of {nbytes}")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s, nb in ((stream, nbytes), (torch.from_numpy(want).cuda(), want.size)):
        y = uz.sentinel_decode(s, n, stream_bytes=nb, status=status)
        assert int(status.item()) == 0
        assert np.array_equal(W.as_u16(y), xh)
    info = uz.stream_info(stream, nbytes)
    assert info["status"] == 0 and info["format"] == _lib.FORMAT_SENTINEL
    assert info["payload_bytes"] == n + (n + 1) // 2 + m
    return m


def test_codebook_tables_match_oracle(uz, orc):
    x, s = W.workload(2, device="cuda", small=True)
    cb = uz.make_sentinel(uz.calibrate(s))
    exps = orc.calibrate(W.as_u16(s))
    enc, dec, esc = orc.sentinel_luts(exps)
    host = cb.cpu().numpy()
    assert np.array_equal(host[48:304], enc) and np.array_equal(host[32:48], dec)
    assert np.array_equal(host[304:560], esc)
    assert host[4] == 2  # the blob's version marks sentinel tables
    rng = np.random.default_rng(6)
    for _ in range(8):
        e = rng.choice(256, 16, replace=False).astype(np.uint8)
        enc, dec, esc = orc.sentinel_luts(e)
        host = sentinel_codebook(uz, e).cpu().numpy()
        assert np.array_equal(host[48:304], enc) and np.array_equal(host[32:48], dec)
        assert np.array_equal(host[304:560], esc)


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_workload_small(uz, orc, k):
    x, s = W.workload(k, device="cuda", small=True)
    exps = orc.calibrate(W.as_u16(s))
    check(uz, orc, x, exps, uz.make_sentinel(uz.calibrate(s)), 1024)


EDGE_CHUNKS = [8, 24, 256, 1000, 1024, 8192, 8200, 16384, 63496, 65536]


@pytest.mark.parametrize("chunk", EDGE_CHUNKS)
def test_edge_sizes(uz, orc, chunk):
    rng = np.random.default_rng(chunk)
    sizes = sorted({1, 2, 7, 8, 9, 15, 31, 32, 33, chunk - 1, chunk, chunk + 1, 3 * chunk + 5, 8191, 8192, 8193,
                    2 * 8192 + 9, 65537, 200_003})
    for n in sizes:
        if rng.random() < 0.5:  # random bit patterns: about 94 % escapes
            xh = rng.integers(0, 65536, n).astype(np.uint16)
        else:  # Gaussian bits: few escapes
            xh = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        if rng.random() < 0.5:
            exps = orc.calibrate(xh)
        check(uz, orc, bf16(xh), exps, sentinel_codebook(uz, exps), chunk)


@pytest.mark.parametrize("chunk", [8, 1024, 65536])
def test_degenerate_inputs(uz, orc, chunk):
    n = 3 * 65536 + 11
    cases = {
        "all zero": np.zeros(n, np.uint16),
        "all escape": np.full(n, 0x3F80, np.uint16),
        "all patterns": np.tile(np.arange(65536, dtype=np.uint32).astype(np.uint16), 3)[:n],
        "specials": np.tile(np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F],
                                     np.uint16), n // 8 + 1)[:n],
    }
    for name, xh in cases.items():
        for exps in (np.arange(16, dtype=np.uint8), orc.calibrate(xh)):
            m = check(uz, orc, bf16(xh), exps, sentinel_codebook(uz, exps), chunk)
            if name == "all escape" and exps[0] == 0:
                assert m == n
            if name == "all patterns" and exps[0] == 0:
                # every exponent 256 times per 65536 patterns, 15 of them coded; the tail's exponent is 0
                assert m == 3 * (65536 - 15 * 256)


def test_the_sixteenth_exponent_escapes(uz, orc):
    """The one exponent that Top-16 codes and Top-15 does not: every one of its
    values becomes an escape of one byte."""
    exps = np.arange(16, dtype=np.uint8) + 100
    xh = np.full(100_003, (115 << 7) | 0x15, np.uint16)  # exponent 115 = exps[15]
    xh[::7] = (100 << 7) | 3
    m = check(uz, orc, bf16(xh), exps, sentinel_codebook(uz, exps), 1024)
    assert m == xh.size - xh[::7].size


def test_empty_input(uz, orc):
    exps = np.arange(16, dtype=np.uint8)
    cb = sentinel_codebook(uz, exps)
    x = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    for chunk in (8, 1024, 65536):
        rc, want = orc.sentinel_encode(np.zeros(0, np.uint16), exps, chunk)
        stream, nbytes = uz.sentinel_encode(x, cb, chunk)
        assert nbytes == want.size == 80
        assert np.array_equal(stream[:nbytes].cpu().numpy(), want)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        uz.sentinel_decode(stream, 0, stream_bytes=nbytes, status=status)
        assert int(status.item()) == 0


def _offsets(stream):
    n = int.from_bytes(stream[8:16].tobytes(), "little")
    chunk = int.from_bytes(stream[16:20].tobytes(), "little")
    nc = -(-n // chunk)
    off_c = 64 + -(-n // 16) * 16 + -(-((n + 1) // 2) // 16) * 16
    return off_c, nc


@pytest.mark.parametrize("chunk", [1024, 65536])
def test_corrupt_streams_are_refused(uz, orc, chunk):
    rng = np.random.default_rng(11)
    n = 5 * 65536 + 17
    xh = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    xh[rng.integers(0, n, 3000)] = 0x7F80  # escapes in every chunk
    exps = orc.calibrate(xh)
    rc, good = orc.sentinel_encode(xh, exps, chunk)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def refused(bad):
        assert orc.sentinel_decode(bad, n)[0] != 0
        status.zero_()
        uz.sentinel_decode(torch.from_numpy(bad).cuda(), n, status=status)
        return int(status.item()) == _lib.ERR_CORRUPT

    for off, flip in ((0, 0xFF), (4, 2), (6, 1), (16, 7), (24, 4), (48, 0x78)):  # magic .. total
        bad = good.copy()
        bad[off] ^= flip
        assert refused(bad), off
    off_c, nc = _offsets(good)
    offs = good[off_c:off_c + 4 * (nc + 1)].view("<u4")
    # one chunk's offset moved down by one: the chunk before it holds one escape more than its values
    bad = good.copy()
    bad[off_c:off_c + 4 * (nc + 1)].view("<u4")[2] = offs[2] - 1
    assert refused(bad)
    # a whole stream decoded as a different length
    status.zero_()
    uz.sentinel_decode(torch.from_numpy(good).cuda(), n + 1, status=status)
    assert int(status.item()) == _lib.ERR_CORRUPT
    # a BF16 Top-16 stream is not a sentinel stream and the other way round
    x = bf16(xh)
    s16, n16 = uz.encode(x, uz.codebook_from_exps(exps.tolist()), chunk)
    status.zero_()
    uz.sentinel_decode(s16, n, stream_bytes=n16, status=status)
    assert int(status.item()) == _lib.ERR_CORRUPT
    status.zero_()
    uz.decode(torch.from_numpy(good).cuda(), n, status=status)
    assert int(status.item()) == _lib.ERR_CORRUPT


@pytest.mark.parametrize("chunk", [8, 1000, 1024, 8200, 65536])
def test_refused_exactly_when_the_oracle_refuses(uz, orc, chunk):
    """Random damage to the header, the offsets and the codes: the GPU status
    equals the oracle's, and where both accept, the values are equal."""
    rng = np.random.default_rng(chunk + 1)
    n = 3 * 65536 + 1001
    xh = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    xh[rng.integers(0, n, 2000)] = 0x7F80
    exps = orc.calibrate(xh)
    rc, good = orc.sentinel_encode(xh, exps, chunk)
    off_c, nc = _offsets(good)
    off_b = 64 + -(-n // 16) * 16
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    refusals = 0
    for trial in range(60):
        bad = good.copy()
        kind = trial % 4
        if kind == 0:  # one offset moved
            j = int(rng.integers(0, nc + 1))
            o = bad[off_c:off_c + 4 * (nc + 1)].view("<u4")
            o[j] = max(0, int(o[j]) + int(rng.choice([-2, -1, 1, 2])))
        elif kind == 1:  # a code turned into 15 or a 15 into another code
            i = int(rng.integers(0, n))
            b = off_b + i // 2
            sh = 4 * (i % 2)
            code = (bad[b] >> sh) & 15
            new = int(rng.integers(0, 15)) if code == 15 else 15
            bad[b] = (bad[b] & (0xF0 >> sh)) | (new << sh)
        elif kind == 2:  # a random byte of codes or offsets
            j = int(rng.integers(off_b, good.size - int.from_bytes(good[24:32].tobytes(), "little")))
            bad[j] ^= np.uint8(1 << int(rng.integers(0, 8)))
        else:  # a random header byte
            j = int(rng.integers(0, 64))
            bad[j] ^= np.uint8(1 << int(rng.integers(0, 8)))
        orc_rc, want = orc.sentinel_decode(bad, n)
        status.zero_()
        y = uz.sentinel_decode(torch.from_numpy(bad).cuda(), n, status=status)
        got = int(status.item())
        assert (got == 0) == (orc_rc == 0), (trial, kind, got, orc_rc)
        if got == 0:
            assert np.array_equal(W.as_u16(y), want), trial
        else:
            refusals += 1
    assert refusals >= 20


def test_code_count_mismatch_inside_a_tile(uz, orc):
    """A chunk that lies inside one decode tile and holds more code 15s than
    its offsets give values is refused."""
    n = 4 * 8192
    xh = np.full(n, 0x3F80, np.uint16)  # exponent 127
    exps = np.arange(16, dtype=np.uint8) + 120  # 127 coded as 7
    rc, good = orc.sentinel_encode(xh, exps, 1024)
    assert int.from_bytes(good[24:32].tobytes(), "little") == 0
    bad = good.copy()
    off_b = 64 + n
    bad[off_b + 600] = 0xF7  # value 1201 of chunk 1 now a code 15, no escape byte for it
    assert orc.sentinel_decode(bad, n)[0] != 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    uz.sentinel_decode(torch.from_numpy(bad).cuda(), n, status=status)
    assert int(status.item()) == _lib.ERR_CORRUPT


def test_stream_copy_moves_sentinel_streams(uz, orc):
    x, s = W.workload(2, device="cuda", small=True)
    cb = uz.make_sentinel(uz.calibrate(s))
    stream, nbytes = uz.sentinel_encode(x, cb, 1024)
    dst = torch.zeros_like(stream)
    copied = torch.zeros(1, dtype=torch.int64, device="cuda")
    uz.stream_copy(stream, dst, copied=copied)
    assert int(copied.item()) == nbytes
    assert torch.equal(dst[:nbytes], stream[:nbytes]) and not dst[nbytes:].any()


def test_kv_full(uz, orc):
    x, s = W.workload(2, device="cuda")
    cb = uz.make_sentinel(uz.calibrate(s))
    exps = orc.calibrate(W.as_u16(s))
    m = check(uz, orc, x, exps, cb, 1024)
    assert m / x.numel() < 0.02
    del x
    torch.cuda.empty_cache()
