"""The BF16 and FP8 E5M2 decoders refuse a stream exactly when the oracle
does (SplitZip review page, §3.2: decode, then the sparse escape overwrite;
§4.1: the round trip is verified bit for bit first). Random damage to the
header, the offsets, the escape positions and values, and the codes: the GPU
status word is UZIP_OK exactly when the oracle accepts, and where both accept,
the decoded values are equal. Integer work: the tolerance is zero."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu


def pad16(v):
    return -(-v // 16) * 16


def _sections(stream, n, chunk, a_bytes):
    nc = -(-n // chunk)
    off_b = 64 + pad16(a_bytes)
    off_c = off_b + pad16(-(-n // 2))
    off_d = off_c + pad16(4 * (nc + 1))
    return nc, off_b, off_c, off_d


def _damage(rng, good, n, chunk, a_bytes, kind):
    """One random change of the kind named; the changed stream may or may not
    still keep the format's rules (the oracle decides)."""
    bad = good.copy()
    nc, off_b, off_c, off_d = _sections(good, n, chunk, a_bytes)
    offs = good[off_c:off_c + 4 * (nc + 1)].view("<u4")
    m = int(offs[nc])
    if kind == 0:  # one offset moved (offsets[0] and offsets[nc] included)
        j = int(rng.choice([0, nc, int(rng.integers(0, nc + 1))]))
        o = bad[off_c:off_c + 4 * (nc + 1)].view("<u4")
        o[j] = max(0, int(o[j]) + int(rng.choice([-2, -1, 1, 2])))
    elif kind in (1, 2):  # a position of a chunk with two or more escapes
        k = np.diff(offs.astype(np.int64))
        cs = np.flatnonzero(k >= 2)
        c = int(rng.choice(cs))
        blk = off_d + 3 * int(offs[c])
        pos = bad[blk:blk + 2 * int(k[c])].view("<u2")
        j = int(rng.integers(1, int(k[c])))
        if kind == 1:  # equal to its neighbour, or one step either way
            pos[j] = max(0, min(65535, int(pos[j - 1]) + int(rng.choice([0, 0, -1, 1]))))
        else:  # two neighbours swapped
            pos[j - 1], pos[j] = int(pos[j]), int(pos[j - 1])
    elif kind == 3:  # a random bit of the escape section
        j = int(rng.integers(off_d, off_d + 3 * m))
        bad[j] ^= np.uint8(1 << int(rng.integers(0, 8)))
    elif kind == 4:  # a random bit of the codes or the offsets
        j = int(rng.integers(off_b, off_d))
        bad[j] ^= np.uint8(1 << int(rng.integers(0, 8)))
    else:  # a random header bit
        j = int(rng.integers(0, 64))
        bad[j] ^= np.uint8(1 << int(rng.integers(0, 8)))
    return bad


def _gauss(rng, n):
    return (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_input(rng, n):
    xh = _gauss(rng, n)
    xh[rng.integers(0, n, n // 50)] = 0x7F80  # +Inf: an escape for an N(0, 1) codebook
    xh[rng.integers(0, n, n // 200)] = 0x0001  # min subnormal: exponent 0
    return xh


@pytest.mark.parametrize("chunk", [64, 1024, 8200])
def test_bf16_refused_exactly_when_the_oracle_refuses(uz, orc, chunk):
    rng = np.random.default_rng(chunk + 11)
    n = 3 * 8192 + 1001 if chunk < 1024 else 3 * 65536 + 1001
    xh = _bf16_input(rng, n)
    exps = orc.calibrate(_gauss(rng, 1 << 16))  # N(0, 1): Inf and exponent 0 escape
    rc, good = orc.encode(xh, exps, chunk)
    assert rc == 0
    assert orc.decode(good, n)[0] == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    refusals = accepted_changed = 0
    for trial in range(72):
        kind = trial % 6
        bad = _damage(rng, good, n, chunk, n, kind)
        orc_rc, want = orc.decode(bad, n)
        status.fill_(-1)
        y = uz.decode(torch.from_numpy(bad).cuda(), n, status=status)
        got = int(status.item())
        assert got in (0, _lib.ERR_CORRUPT), (trial, kind, got)
        assert (got == 0) == (orc_rc == 0), (trial, kind, got, orc_rc)
        if got == 0:
            assert np.array_equal(W.as_u16(y), want), (trial, kind)
            accepted_changed += not np.array_equal(want, xh)
        else:
            refusals += 1
    assert refusals >= 30 and accepted_changed >= 5


@pytest.mark.parametrize("chunk", [64, 1024])
def test_e5m2_refused_exactly_when_the_oracle_refuses(uz, orc, chunk):
    rng = np.random.default_rng(chunk + 12)
    n = 2 * 16384 + 999 if chunk < 1024 else 3 * 65536 + 999
    x = rng.integers(0, 256, n).astype(np.uint8)
    x[rng.random(n) < 0.6] = 0x3C  # 1.0: a skewed law, so the codebook leaves escapes
    exps = orc.e5m2_calibrate(x[: n // 2])
    rc, good = orc.e5m2_encode(x, exps, chunk)
    assert rc == 0
    a_bytes = 3 * (-(-n // 8))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    refusals = 0
    for trial in range(60):
        kind = trial % 6
        bad = _damage(rng, good, n, chunk, a_bytes, kind)
        orc_rc, want = orc.e5m2_decode(bad, n)
        status.fill_(-1)
        y = uz.e5m2_decode(torch.from_numpy(bad).cuda(), n, status=status)
        got = int(status.item())
        assert got in (0, _lib.ERR_CORRUPT), (trial, kind, got)
        assert (got == 0) == (orc_rc == 0), (trial, kind, got, orc_rc)
        if got == 0:
            assert np.array_equal(W.as_u8(y), want), (trial, kind)
        else:
            refusals += 1
    assert refusals >= 25


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_offsets_span_and_repeated_positions(uz, orc, fmt):
    """The cases the decoders used to accept: offsets that start above 0 or end
    below M with every other rule kept, and a repeated position in a block."""
    rng = np.random.default_rng(5)
    n, chunk = 4 * 8192 + 77, 256
    if fmt == "bf16":
        x = _bf16_input(rng, n)
        exps = orc.calibrate(_gauss(rng, 1 << 16))
        rc, good = orc.encode(x, exps, chunk)
        a_bytes, dec_o, dec_g = n, orc.decode, uz.decode
    else:
        x = rng.integers(0, 256, n).astype(np.uint8)
        x[rng.random(n) < 0.6] = 0x3C
        exps = orc.e5m2_calibrate(x)
        rc, good = orc.e5m2_encode(x, exps, chunk)
        a_bytes, dec_o, dec_g = 3 * (-(-n // 8)), orc.e5m2_decode, uz.e5m2_decode
    assert rc == 0
    nc, off_b, off_c, off_d = _sections(good, n, chunk, a_bytes)
    offs = good[off_c:off_c + 4 * (nc + 1)].view("<u4").astype(np.int64)

    def grown(offsets, lead):  # one more escape slot in the header, three spare bytes
        g = np.concatenate([good[:off_d], np.zeros(3, np.uint8) if lead else good[off_d:],
                            good[off_d:] if lead else np.zeros(3, np.uint8)])
        g[24:32] = np.frombuffer(np.uint64(offs[nc] + 1).tobytes(), np.uint8)
        g[48:56] = np.frombuffer(np.uint64(g.size).tobytes(), np.uint8)
        g[off_c:off_c + 4 * (nc + 1)] = np.frombuffer(offsets.astype("<u4").tobytes(), np.uint8)
        return g

    c = int(np.flatnonzero(np.diff(offs) >= 2)[-1])  # the last chunk with two escapes or more
    rep = good.copy()
    blk = off_d + 3 * int(offs[c])
    rep[blk + 2:blk + 4] = rep[blk:blk + 2]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (grown(offs + 1, True), grown(offs, False), rep):
        assert dec_o(bad, n)[0] != 0
        status.zero_()
        dec_g(torch.from_numpy(bad).cuda(), n, status=status)
        assert int(status.item()) == _lib.ERR_CORRUPT
    # the good stream is still accepted
    status.fill_(-1)
    dec_g(torch.from_numpy(good).cuda(), n, status=status)
    assert int(status.item()) == 0


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_empty_stream_offsets(uz, orc, fmt):
    """n = 0: the single offset must be 0."""
    if fmt == "bf16":
        rc, good = orc.encode(np.zeros(0, np.uint16), np.arange(16, dtype=np.uint8), 1024)
        dec_o, dec_g = orc.decode, uz.decode
    else:
        rc, good = orc.e5m2_encode(np.zeros(0, np.uint8), np.arange(16, dtype=np.uint8), 1024)
        dec_o, dec_g = orc.e5m2_decode, uz.e5m2_decode
    assert rc == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for v, ok in ((0, True), (1, False)):
        s = good.copy()
        s[64 + 0] = v  # offsets[0] sits right after the header when n = 0
        assert (dec_o(s, 0)[0] == 0) == ok
        status.fill_(-1)
        dec_g(torch.from_numpy(s).cuda(), 0, status=status)
        assert (int(status.item()) == 0) == ok
