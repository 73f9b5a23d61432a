"""Pins for the oracle's FP8 E5M2 variant (SplitZip review page, §4.2 and
appendix C: the Top-16 framework applied to E5M2 KV values, a further 1.14x),
each against something other than the oracle itself:

  - the split against the numeric meaning of every one of the 256 patterns
    (an E5M2 byte is the high byte of an IEEE-754 binary16 value, so numpy's
    float16 fixes sign, exponent and mantissa);
  - a complete stream worked out by hand (tests/golden/stream_e5m2_n10_chunk8.txt);
  - closed forms: payload 3 ceil(n/8) + ceil(n/2) + 3M, the 8/7 ratio with no
    escapes, exactly half of an all-patterns tensor escaping for any codebook;
  - every section of brute-force tiny streams read back with numpy;
  - corrupt streams refused.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL = np.arange(256, dtype=np.uint8)


def fp16_fields(x):
    """(exponent field, sign, 2-bit mantissa) of E5M2 bytes from the value of
    the binary16 number whose high byte they are."""
    h = (x.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    sign = np.signbit((x.astype(np.uint16) << 8).view(np.float16)).astype(np.uint8)
    e = np.zeros(x.size, np.uint8)
    m = np.zeros(x.size, np.uint8)
    for i, v in enumerate(h):
        a = abs(v)
        if np.isnan(v) or np.isinf(v):
            e[i] = 31
            m[i] = x[i] & 3 if np.isnan(v) else 0  # NaN payload: the pattern's own bits
        elif a < 2.0 ** -14:  # zero and subnormals: value = m / 4 * 2^-14
            e[i] = 0
            m[i] = int(round(a / 2.0 ** -14 * 4))
        else:
            k = int(np.floor(np.log2(a)))
            e[i] = k + 15
            m[i] = int(round((a / 2.0 ** k - 1) * 4))
    return e, sign, m


def test_split_matches_binary16_semantics(orc):
    e, a = orc.e5m2_split(ALL)
    fe, fs, fm = fp16_fields(ALL)
    assert np.array_equal(e, fe)
    assert np.array_equal(a >> 2, fs)
    assert np.array_equal(a & 3, fm)
    assert e.max() == 31 and a.max() == 7


def test_merge_inverts_split_and_is_a_bijection(orc):
    e, a = orc.e5m2_split(ALL)
    assert np.array_equal(orc.e5m2_merge(a, e), ALL)
    ee, aa = np.meshgrid(np.arange(32, dtype=np.uint8), np.arange(8, dtype=np.uint8))
    x = orc.e5m2_merge(aa.ravel(), ee.ravel())
    assert np.unique(x).size == 256


def test_histogram_and_top16(orc):
    rng = np.random.default_rng(3)
    x = rng.integers(0, 256, 5000).astype(np.uint8)
    fe = fp16_fields(x)[0]
    h = orc.e5m2_histogram(x)
    assert np.array_equal(h[:32], np.bincount(fe, minlength=32)) and not h[32:].any()
    # two exponents only: most frequent first, then unseen ones in ascending order
    x = np.array([0x0C] * 5 + [0x1C] * 9, np.uint8)  # exponents 3 (x5) and 7 (x9)
    exps = orc.e5m2_calibrate(x)
    assert exps.tolist() == [7, 3, 0, 1, 2, 4, 5, 6, 8, 9, 10, 11, 12, 13, 14, 15]
    # ties: smaller exponent first
    x = np.array([0x10, 0x10, 0x08, 0x08], np.uint8)  # exponents 4 and 2, twice each
    assert orc.e5m2_calibrate(x)[:2].tolist() == [2, 4]


def _golden():
    exps, x, stream, chunk = None, None, [], None
    with open(os.path.join(GOLDEN, "stream_e5m2_n10_chunk8.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "exps":
                exps = np.array([int(v, 16) for v in vals], np.uint8)
            elif key == "x":
                x = np.array([int(v, 16) for v in vals], np.uint8)
            elif key == "chunk":
                chunk = int(vals[0])
            elif key == "stream":
                stream += [int(v, 16) for v in vals]
    return exps, x, chunk, np.array(stream, np.uint8)


def test_encode_matches_hand_worked_stream(orc):
    exps, x, chunk, want = _golden()
    rc, got = orc.e5m2_encode(x, exps, chunk)
    assert rc == oracle.OK
    assert got.tobytes().hex() == want.tobytes().hex()
    rc, back = orc.e5m2_decode(want, x.size)
    assert rc == oracle.OK and np.array_equal(back, x)


def pad16(v):
    return (v + 15) // 16 * 16


def check_e5m2_stream(stream, x, exps, chunk):
    """Read an E5M2 stream section by section with numpy against the format."""
    n = x.size
    nc = -(-n // chunk)
    fe, fs, fm = fp16_fields(x)
    esc = ~np.isin(fe, exps)
    m = int(esc.sum())
    off_a = 64
    off_b = off_a + pad16(3 * (-(-n // 8)))
    off_c = off_b + pad16(-(-n // 2))
    off_d = off_c + pad16(4 * (nc + 1))
    assert stream.size == off_d + 3 * m
    h = stream[:64]
    assert h[:4].tobytes() == b"UZE1" and h[4] == 1 and h[5:8].sum() == 0
    assert int.from_bytes(h[8:16].tobytes(), "little") == n
    assert int.from_bytes(h[24:32].tobytes(), "little") == m
    assert np.array_equal(h[32:48], exps) and int.from_bytes(h[48:56].tobytes(), "little") == stream.size
    # A: fields from the words
    groups = -(-n // 8)
    A = stream[off_a:off_a + 3 * groups].astype(np.uint32).reshape(groups, 3)
    words = A[:, 0] | (A[:, 1] << 8) | (A[:, 2] << 16)
    fields = ((words[:, None] >> (3 * np.arange(8))) & 7).reshape(-1)
    assert np.array_equal(fields[:n], (fs << 2) | fm) and not fields[n:].any()
    assert not stream[off_a + 3 * groups:off_b].any()
    # B: codes (escapes 0)
    lut = np.zeros(32, np.uint8)
    lut[exps] = np.arange(16)
    codes = np.where(esc, 0, lut[fe])
    B = stream[off_b:off_b + -(-n // 2)]
    got = np.stack([B & 15, B >> 4], 1).reshape(-1)
    assert np.array_equal(got[:n], codes) and (n % 2 == 0 or got[n] == 0)
    # C and D
    idx = np.flatnonzero(esc)
    per = np.bincount(idx // chunk, minlength=nc)
    offs = stream[off_c:off_c + 4 * (nc + 1)].view("<u4")
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(per)]))
    D = stream[off_d:]
    for c in range(nc):
        o, k = int(offs[c]), int(per[c])
        mine = idx[(idx >= c * chunk) & (idx < (c + 1) * chunk)]
        pos = D[3 * o:3 * o + 2 * k].view("<u2")
        assert np.array_equal(pos, mine - c * chunk)
        assert np.array_equal(D[3 * o + 2 * k:3 * o + 3 * k], fe[mine])
    return m


@pytest.mark.parametrize("chunk", [8, 16, 24, 64, 1024])
def test_brute_force_tiny_streams(orc, chunk):
    rng = np.random.default_rng(chunk)
    for n in sorted({0, 1, 2, 7, 8, 9, chunk - 1, chunk, chunk + 1, 3 * chunk + 5}):
        x = rng.integers(0, 256, n).astype(np.uint8)
        exps = rng.choice(32, 16, replace=False).astype(np.uint8)
        rc, s = orc.e5m2_encode(x, exps, chunk)
        assert rc == oracle.OK
        check_e5m2_stream(s, x, exps, chunk)
        rc, y = orc.e5m2_decode(s, n)
        assert rc == oracle.OK and np.array_equal(y, x)


def test_closed_forms(orc):
    # no escapes: exactly 7 bits per value, ratio 8/7 (the page's 1.14x)
    n = 8 * 4096
    x = np.full(n, 0x3C, np.uint8)
    exps = orc.e5m2_calibrate(x)
    rc, s = orc.e5m2_encode(x, exps, 1024)
    payload = 3 * (n // 8) + n // 2
    assert Fraction(n, payload) == Fraction(8, 7)
    assert s.size == orc.e5m2_stream_bytes(n, 0, 1024)
    # all 256 patterns, any codebook: every exponent 8 times, 16 of 32 escape
    x = np.tile(ALL, 5)
    for seed in range(4):
        exps = np.random.default_rng(seed).choice(32, 16, replace=False).astype(np.uint8)
        rc, s = orc.e5m2_encode(x, exps, 256)
        m = int.from_bytes(s[24:32].tobytes(), "little")
        assert m == x.size // 2
        assert s.size == orc.e5m2_stream_bytes(x.size, m, 256)
        rc, y = orc.e5m2_decode(s, x.size)
        assert np.array_equal(y, x)


def test_corrupt_streams_are_refused(orc):
    exps, x, chunk, good = _golden()
    assert orc.e5m2_decode(good, x.size)[0] == oracle.OK
    for off, val in ((0, 0x00), (4, 2), (6, 1), (8, 11), (16, 7), (24, 4), (48, 0x78)):
        bad = good.copy()
        bad[off] = val
        assert orc.e5m2_decode(bad, x.size)[0] == oracle.ERR_CORRUPT, off
    bad = good.copy()
    bad[112] = 9  # escape position past its chunk of 8
    assert orc.e5m2_decode(bad, x.size)[0] == oracle.ERR_CORRUPT
    # offsets (at 96) must run from 0 to M; chunk 0's positions (4, 5 at 112)
    # must rise strictly, one entry per escape
    for edits in ({96: 1}, {104: 2}, {114: 4}, {112: 5, 114: 4}):
        bad = good.copy()
        for k, v in edits.items():
            bad[k] = v
        assert orc.e5m2_decode(bad, x.size)[0] == oracle.ERR_CORRUPT, edits
    assert orc.e5m2_decode(good, x.size - 1)[0] == oracle.ERR_CORRUPT
    # a BF16 stream is not an E5M2 stream
    assert orc.e5m2_decode(orc.encode(np.zeros(10, np.uint16), np.arange(16), 8)[1], 10)[0] == oracle.ERR_CORRUPT
