"""Pins for the oracle's Top-15 + sentinel variant (SplitZip review page,
§3.4 and §4.3 Table 6: code 15 marks an escape, no positions stored), each
against something other than the oracle: a stream worked out by hand, the
closed-form size, the coverage relation with the Top-16 codec, brute-force
section reads, corrupt streams."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    exps, x, stream, chunk = None, None, [], None
    with open(os.path.join(GOLDEN, "stream_sentinel_n10_chunk8.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "exps":
                exps = np.array([int(v, 16) for v in vals], np.uint8)
            elif key == "x":
                x = np.array([int(v, 16) for v in vals], np.uint16)
            elif key == "chunk":
                chunk = int(vals[0])
            elif key == "stream":
                stream += [int(v, 16) for v in vals]
    return exps, x, chunk, np.array(stream, np.uint8)


def ieee_exponent(x):
    """Exponent field of BF16 patterns from the float32 value they widen to."""
    f = (x.astype(np.uint32) << 16).view(np.float32)
    return ((f.view(np.uint32) >> 23) & 0xFF).astype(np.uint8)


def test_encode_matches_hand_worked_stream(orc):
    exps, x, chunk, want = _golden()
    exps16 = np.concatenate([exps, [0x87]]).astype(np.uint8)  # the 16th entry is not used
    rc, got = orc.sentinel_encode(x, exps16, chunk)
    assert rc == oracle.OK
    assert got.tobytes().hex() == want.tobytes().hex()
    rc, back = orc.sentinel_decode(want, x.size)
    assert rc == oracle.OK and np.array_equal(back, x)


def test_luts(orc):
    rng = np.random.default_rng(2)
    for _ in range(10):
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        enc, dec, esc = orc.sentinel_luts(exps)
        assert np.array_equal(enc[exps[:15]], np.arange(15)) and np.array_equal(dec[:15], exps[:15])
        outside = ~np.isin(np.arange(256), exps[:15])
        assert np.all(enc[outside] == 15) and np.array_equal(esc.astype(bool), outside)


def check_sentinel_stream(s, x, exps, chunk):
    n = x.size
    nc = -(-n // chunk)
    e = ieee_exponent(x)
    esc = ~np.isin(e, exps[:15])
    m = int(esc.sum())
    pad = lambda v: (v + 15) // 16 * 16
    off_b = 64 + pad(n)
    off_c = off_b + pad(-(-n // 2))
    off_d = off_c + pad(4 * (nc + 1))
    assert s.size == off_d + m  # n + ceil(n/2) + M payload, one byte per escape
    assert s[:4].tobytes() == b"UZS1" and np.array_equal(s[32:47], exps[:15]) and s[47] == 0
    lut = np.full(256, 15, np.uint8)
    lut[exps[:15]] = np.arange(15)
    B = s[off_b:off_b + -(-n // 2)]
    codes = np.stack([B & 15, B >> 4], 1).reshape(-1)[:n]
    assert np.array_equal(codes, lut[e]) and np.array_equal(codes == 15, esc)
    offs = s[off_c:off_c + 4 * (nc + 1)].view("<u4")
    per = np.bincount(np.flatnonzero(esc) // chunk, minlength=nc)
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(per)]))
    assert np.array_equal(s[off_d:], e[esc])  # values in ascending element order
    return m


@pytest.mark.parametrize("chunk", [8, 24, 1024])
def test_brute_force_tiny_streams(orc, chunk):
    rng = np.random.default_rng(chunk)
    for n in sorted({0, 1, 2, 7, 8, 9, chunk - 1, chunk, chunk + 1, 3 * chunk + 5}):
        x = rng.integers(0, 65536, n).astype(np.uint16)
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        rc, s = orc.sentinel_encode(x, exps, chunk)
        assert rc == oracle.OK
        check_sentinel_stream(s, x, exps, chunk)
        rc, y = orc.sentinel_decode(s, n)
        assert rc == oracle.OK and np.array_equal(y, x)


def test_closed_forms_and_coverage(orc):
    # all 65536 patterns: each exponent 256 times, 15 in the codebook
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exps = np.random.default_rng(5).choice(256, 16, replace=False).astype(np.uint8)
    rc, s = orc.sentinel_encode(x, exps, 1024)
    m = int.from_bytes(s[24:32].tobytes(), "little")
    assert m == 65536 - 15 * 256 and s.size == orc.sentinel_stream_bytes(65536, m, 1024)
    # against the Top-16 codec: one exponent fewer in the codebook, one byte per escape instead of three
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(100_000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    exps = orc.calibrate(x)
    m16 = orc.count_escapes(x, exps)
    rc, s = orc.sentinel_encode(x, exps, 1024)
    m15 = int.from_bytes(s[24:32].tobytes(), "little")
    assert m15 - m16 == int(np.sum(ieee_exponent(x) == exps[15]))
    rc, s16 = orc.encode(x, exps, 1024)
    assert s16.size - s.size == 3 * m16 - m15


def test_corrupt_streams_are_refused(orc):
    exps, x, chunk, good = _golden()
    exps16 = np.concatenate([exps, [0x87]]).astype(np.uint8)
    assert orc.sentinel_decode(good, x.size)[0] == oracle.OK
    for off, val in ((0, 0), (4, 2), (6, 1), (8, 11), (16, 7), (24, 4), (48, 0x72)):
        bad = good.copy()
        bad[off] = val
        assert orc.sentinel_decode(bad, x.size)[0] == oracle.ERR_CORRUPT, off
    bad = good.copy()
    bad[80] = 0xF0  # a fourth code 15 in chunk 0: more escapes than values
    assert orc.sentinel_decode(bad, x.size)[0] == oracle.ERR_CORRUPT
    bad = good.copy()
    bad[81] = 0x02  # one code 15 fewer: a value left over
    assert orc.sentinel_decode(bad, x.size)[0] == oracle.ERR_CORRUPT
    assert orc.sentinel_decode(orc.encode(x, exps16, chunk)[1], x.size)[0] == oracle.ERR_CORRUPT
