"""Pins of the CPU oracle against what the SplitZip review page and mathematics
fix, independent of the oracle's own formulas:

- the bit split (§3.2) against IEEE-754 semantics of the BF16 value (numpy's
  float32 frexp / signbit), exhaustively over all 65,536 patterns, and against
  hand-worked examples;
- the histogram (§3.3) against numpy's bincount of those IEEE exponents;
- the Top-16 choice (§3.3) against maximal coverage and hand-built tie cases;
- the stream (§3.2) against a hand-worked complete stream, the page's closed
  form N + N/2 + 3M and rho = 2 / (3/2 + 3 eps), its 4/3 limit, and a
  section-by-section reading of the bytes with numpy set operations;
- decode(encode(x)) == x on tiny brute-force cases and special values.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


# ----------------------------------------------------------- IEEE semantics

def ieee_fields(x16):
    """(biased exponent, sign bit, 7-bit mantissa) of BF16 patterns, derived
    from the float value (not from shifts of the pattern)."""
    x16 = np.asarray(x16, np.uint16)
    v32 = (x16.astype(np.uint32) << 16).view(np.float32)
    sign = np.signbit(v32).astype(np.uint8)
    with np.errstate(invalid="ignore"):
        v = v32.astype(np.float64)
    av = np.abs(v)
    e = np.zeros(v.shape, np.int64)
    mant = np.zeros(v.shape, np.int64)
    finite = np.isfinite(v)
    normal = finite & (av >= 2.0 ** -126)
    sub = finite & (av > 0) & (av < 2.0 ** -126)
    m, k = np.frexp(av[normal])  # av = m * 2**k, m in [0.5, 1)
    e[normal] = k + 126
    frac = (m * 2 - 1) * 128
    assert np.all(frac == np.round(frac))
    mant[normal] = frac.astype(np.int64)
    q = av[sub] / 2.0 ** -133  # subnormal step of BF16
    assert np.all(q == np.round(q))
    mant[sub] = q.astype(np.int64)
    e[~finite] = 255
    nan = np.isnan(v32)
    # A NaN has no numeric mantissa: its payload is the stored field itself.
    # Infinity has mantissa 0 (left at zero above).
    mant[nan] = (x16[nan] & 0x7F).astype(np.int64)
    return e.astype(np.uint8), sign, mant.astype(np.uint8)


def ieee_a(x16):
    _, s, m = ieee_fields(x16)
    return ((s << 7) | m).astype(np.uint8)


# ------------------------------------------------------------------- split

def test_split_hand_worked_examples(orc):
    rows = []
    with open(os.path.join(GOLDEN, "bit_split.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                x, e, a, _ = line.split(None, 3)
                rows.append((int(x, 16), int(e, 16), int(a, 16)))
    x = np.array([r[0] for r in rows], np.uint16)
    e, a = orc.split(x)
    assert e.tolist() == [r[1] for r in rows]
    assert a.tolist() == [r[2] for r in rows]
    assert orc.merge(a, e).tolist() == x.tolist()


def test_split_matches_ieee_fields_exhaustively(orc):
    e, a = orc.split(ALL)
    ie, isign, imant = ieee_fields(ALL)
    assert np.array_equal(e, ie)
    assert np.array_equal(a >> 7, isign)
    assert np.array_equal(a & 0x7F, imant)


def test_merge_is_a_bijection_inverse_of_split(orc):
    e, a = orc.split(ALL)
    assert np.array_equal(orc.merge(a, e), ALL)
    # every (a, e) pair is hit exactly once
    pair = a.astype(np.uint32) << 8 | e
    assert np.unique(pair).size == 65536
    # and merge of every pair lands on a distinct pattern
    aa, ee = np.meshgrid(np.arange(256, dtype=np.uint8), np.arange(256, dtype=np.uint8))
    xs = orc.merge(aa.reshape(-1), ee.reshape(-1))
    assert np.unique(xs).size == 65536
    e2, a2 = orc.split(xs)
    assert np.array_equal(e2, ee.reshape(-1)) and np.array_equal(a2, aa.reshape(-1))


# ------------------------------------------------------------- calibration

def test_histogram_is_bincount_of_ieee_exponents(orc):
    rng = np.random.default_rng(7)
    x = rng.integers(0, 65536, 100_003).astype(np.uint16)
    ie, _, _ = ieee_fields(x)
    assert np.array_equal(orc.histogram(x), np.bincount(ie, minlength=256).astype(np.uint64))
    assert int(orc.histogram(x).sum()) == x.size


def _hist(pairs):
    h = np.zeros(256, np.uint64)
    for v, c in pairs:
        h[v] = c
    return h


@pytest.mark.parametrize(
    "pairs, expect",
    [
        # all zero: nothing seen, codes fill in ascending exponent order
        ([], list(range(16))),
        # three seen exponents, two of them tied: tie -> smaller value first,
        # unseen exponents then fill in ascending order skipping the seen ones
        ([(200, 5), (100, 7), (7, 5)], [100, 7, 200, 0, 1, 2, 3, 4, 5, 6, 8, 9, 10, 11, 12, 13]),
        # 20 distinct counts: the 16 largest, most frequent first
        ([(v, 1000 - 10 * i) for i, v in enumerate(range(110, 130))], list(range(110, 126))),
        # tie exactly at the cut: exponents 50 and 40 both have the 16th count
        ([(v, 100 + v) for v in range(60, 75)] + [(50, 3), (40, 3)],
         list(range(74, 59, -1)) + [40]),
    ],
)
def test_top16_hand_built(orc, pairs, expect):
    assert orc.top16(_hist(pairs)).tolist() == expect


def test_top16_has_maximal_coverage(orc):
    rng = np.random.default_rng(11)
    for _ in range(50):
        h = rng.integers(0, 50, 256).astype(np.uint64) * rng.integers(0, 2, 256).astype(np.uint64)
        exps = orc.top16(h)
        assert np.unique(exps).size == 16
        assert int(h[exps].sum()) == int(np.sort(h)[-16:].sum())
        counts = h[exps].astype(np.int64)
        assert np.all(np.diff(counts) <= 0)  # most frequent first


def test_luts_are_consistent_with_codebook(orc):
    rng = np.random.default_rng(3)
    for _ in range(20):
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        enc, dec, esc = orc.luts(exps)
        assert np.array_equal(dec, exps)
        assert np.array_equal(enc[exps], np.arange(16))
        outside = ~np.isin(np.arange(256), exps)
        assert np.array_equal(esc.astype(bool), outside)
        assert np.all(enc[outside] == 0)  # dummy code


# ------------------------------------------------------------------ stream

def _read_golden_stream():
    exps, x, stream, chunk = None, None, [], None
    with open(os.path.join(GOLDEN, "stream_n10_chunk8.txt")) as f:
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


def test_encode_matches_hand_worked_stream(orc):
    exps, x, chunk, want = _read_golden_stream()
    rc, got = orc.encode(x, exps, chunk)
    assert rc == oracle.OK
    assert got.tobytes().hex() == want.tobytes().hex()
    rc, back = orc.decode(want, x.size)
    assert rc == oracle.OK and np.array_equal(back, x)


def pad16(v):
    return (v + 15) // 16 * 16


def check_stream(stream, x, exps, chunk):
    """Read a version-1 stream section by section with numpy and check each
    part against what the page defines for it."""
    x = np.asarray(x, np.uint16)
    n = x.size
    nc = -(-n // chunk)
    ie = ieee_fields(x)[0]
    escape = ~np.isin(ie, exps)
    m = int(escape.sum())
    hdr = stream[:64].tobytes()
    assert hdr[:4] == b"UZP1"
    assert int.from_bytes(hdr[4:6], "little") == 1 and int.from_bytes(hdr[6:8], "little") == 0
    assert int.from_bytes(hdr[8:16], "little") == n
    assert int.from_bytes(hdr[16:20], "little") == chunk
    assert int.from_bytes(hdr[20:24], "little") == nc
    assert int.from_bytes(hdr[24:32], "little") == m
    assert hdr[32:48] == exps.tobytes()
    off_a, off_b = 64, 64 + pad16(n)
    off_c = off_b + pad16((n + 1) // 2)
    off_d = off_c + pad16(4 * (nc + 1))
    total = off_d + 3 * m
    assert int.from_bytes(hdr[48:56], "little") == total == stream.size
    assert hdr[56:64] == bytes(8)
    # A: exact sign-mantissa bytes, zero padding
    assert np.array_equal(stream[off_a:off_a + n], ieee_a(x))
    assert not stream[off_a + n:off_b].any()
    # B: codes, low nibble first; codebook exponent for hits, dummy 0 for escapes
    packed = stream[off_b:off_b + (n + 1) // 2]
    codes = np.empty(2 * packed.size, np.uint8)
    codes[0::2], codes[1::2] = packed & 0xF, packed >> 4
    if n % 2:
        assert codes[n] == 0
    codes = codes[:n]
    assert np.array_equal(exps[codes[~escape]], ie[~escape])
    assert np.all(codes[escape] == 0)
    assert not stream[off_b + (n + 1) // 2:off_c].any()
    # C: exclusive prefix of per-chunk escape counts
    per_chunk = np.bincount(np.flatnonzero(escape) // chunk, minlength=nc) if nc else np.zeros(0, int)
    want_off = np.concatenate([[0], np.cumsum(per_chunk)]).astype(np.uint32)
    got_off = stream[off_c:off_c + 4 * (nc + 1)].view("<u4")
    assert np.array_equal(got_off, want_off)
    assert not stream[off_c + 4 * (nc + 1):off_d].any()
    # D: per chunk, ascending positions then raw exponents
    D = stream[off_d:]
    for c in range(nc):
        k = int(per_chunk[c])
        blk = D[3 * want_off[c]:3 * want_off[c] + 3 * k]
        where = np.flatnonzero(escape[c * chunk:(c + 1) * chunk])
        assert np.array_equal(blk[:2 * k].view("<u2"), where)
        assert np.array_equal(blk[2 * k:], ie[c * chunk + where])
    return m


def closed_form_check(stream, n, m):
    payload = n + (n + 1) // 2 + 3 * m
    if n and n % 2 == 0:
        eps = Fraction(m, n)
        assert Fraction(payload) == n * (Fraction(3, 2) + 3 * eps)
        assert Fraction(2 * n, payload) == 2 / (Fraction(3, 2) + 3 * eps)
    return payload


def _random_codebook(rng, x):
    """Half the time the calibrated codebook, else 16 random exponents."""
    if rng.random() < 0.5:
        h = np.bincount(ieee_fields(x)[0], minlength=256)
        return np.argsort(-h, kind="stable")[:16].astype(np.uint8)
    return rng.choice(256, 16, replace=False).astype(np.uint8)


@pytest.mark.parametrize("chunk", [8, 16, 24, 256, 1024])
def test_brute_force_tiny_inputs(orc, chunk):
    rng = np.random.default_rng(chunk)
    sizes = sorted({0, 1, 2, 7, 8, 9, chunk - 1, chunk, chunk + 1, 3 * chunk + 5})
    for n in sizes:
        for trial in range(3):
            if trial == 0:
                x = rng.integers(0, 65536, n).astype(np.uint16)
            else:  # Gaussian-like, mostly inside the codebook
                x = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            exps = _random_codebook(rng, x)
            rc, s = orc.encode(x, exps, chunk)
            assert rc == oracle.OK
            m = check_stream(s, x, exps, chunk)
            assert s.size == orc.stream_bytes(n, m, chunk)
            assert m == orc.count_escapes(x, exps)
            closed_form_check(s, n, m)
            rc, back = orc.decode(s, n)
            assert rc == oracle.OK and np.array_equal(back, x)


def test_all_patterns_tensor(orc):
    """Each exponent occurs 256 times among the 65,536 patterns, so any
    codebook leaves 65,536 - 16 * 256 = 61,440 escapes; payload
    65,536 + 32,768 + 3 * 61,440 = 282,624 bytes."""
    rng = np.random.default_rng(5)
    x = rng.permutation(ALL)
    for _ in range(3):
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        rc, s = orc.encode(x, exps, 1024)
        assert rc == oracle.OK
        m = check_stream(s, x, exps, 1024)
        assert m == 61440
        assert closed_form_check(s, x.size, m) == 282624
        rc, back = orc.decode(s, x.size)
        assert rc == oracle.OK and np.array_equal(back, x)


def test_all_zero_reaches_four_thirds(orc):
    """No escape at all: payload is exactly 3/4 of the raw bytes (the 4/3
    asymptote of rho in §3.2)."""
    x = np.zeros(4096, np.uint16)
    exps = orc.calibrate(x)
    assert exps[0] == 0
    rc, s = orc.encode(x, exps, 1024)
    assert rc == oracle.OK
    assert check_stream(s, x, exps, 1024) == 0
    assert Fraction(2 * x.size, closed_form_check(s, x.size, 0)) == Fraction(4, 3)


def test_every_value_an_escape(orc):
    x = np.full(3000, 0x3F80, np.uint16)  # 1.0 -> exponent 0x7F
    exps = np.arange(16, dtype=np.uint8)  # does not contain 0x7F
    rc, s = orc.encode(x, exps, 256)
    assert rc == oracle.OK
    assert check_stream(s, x, exps, 256) == 3000
    rc, back = orc.decode(s, x.size)
    assert rc == oracle.OK and np.array_equal(back, x)


def test_special_values_round_trip(orc):
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F,
                         0x0080, 0x7F7F, 0xFF7F, 0x3F80], np.uint16)
    x = np.tile(specials, 50)
    for exps in (orc.calibrate(x), np.arange(16, dtype=np.uint8)):
        rc, s = orc.encode(x, exps, 8)
        assert rc == oracle.OK
        check_stream(s, x, exps, 8)
        rc, back = orc.decode(s, x.size)
        assert rc == oracle.OK and np.array_equal(back, x)


# ------------------------------------------------------------- error cases

def test_encode_rejects_bad_arguments(orc):
    x = np.zeros(100, np.uint16)
    exps = np.arange(16, dtype=np.uint8)
    for chunk in (0, 4, 12, 65544, 1 << 20):
        assert orc.encode(x, exps, chunk)[0] == oracle.ERR_CHUNK
    need = orc.stream_bytes(100, 0, 64)
    assert orc.encode(x, exps, 64, cap=need - 1)[0] == oracle.ERR_CAPACITY
    assert orc.encode(x, exps, 64, cap=need)[0] == oracle.OK


def test_decode_rejects_corrupt_streams(orc):
    rng = np.random.default_rng(9)
    x = rng.integers(0, 65536, 1000).astype(np.uint16)
    exps = np.arange(120, 136, dtype=np.uint8)
    rc, s = orc.encode(x, exps, 64)
    assert rc == oracle.OK
    assert orc.decode(s, 1000)[0] == oracle.OK
    assert orc.decode(s, 999)[0] == oracle.ERR_CORRUPT            # n mismatch
    assert orc.decode(s[:-1], 1000)[0] == oracle.ERR_CORRUPT      # truncated
    bad = s.copy(); bad[0] ^= 1
    assert orc.decode(bad, 1000)[0] == oracle.ERR_CORRUPT         # magic
    bad = s.copy(); bad[6] = 1
    assert orc.decode(bad, 1000)[0] == oracle.ERR_CORRUPT         # status flag set
    nc = -(-1000 // 64)
    off_c = 64 + pad16(1000) + pad16(500)
    bad = s.copy(); bad[off_c + 4 * 3:off_c + 4 * 4] = np.frombuffer(np.uint32(10**6).tobytes(), np.uint8)
    assert orc.decode(bad, 1000)[0] == oracle.ERR_CORRUPT         # offsets not rising
    off_d = off_c + pad16(4 * (nc + 1))
    bad = s.copy(); bad[off_d:off_d + 2] = [0xFF, 0xFF]
    assert orc.decode(bad, 1000)[0] == oracle.ERR_CORRUPT         # position outside chunk
    offs = s[off_c:off_c + 4 * (nc + 1)].view("<u4").astype(np.int64)
    # Offsets must run from 0 to M. Two streams that break only that rule:
    # one escape slot more in the header (M + 1, total + 3) with three spare
    # bytes before every block and all offsets raised by one (offsets[0] = 1),
    # or after the last block with the offsets unchanged (offsets[nc] = M).
    def grown(offsets, lead):
        m1 = int(offs[nc]) + 1
        g = np.concatenate([s[:off_d], np.zeros(3, np.uint8) if lead else s[off_d:],
                            s[off_d:] if lead else np.zeros(3, np.uint8)])
        g[24:32] = np.frombuffer(np.uint64(m1).tobytes(), np.uint8)
        g[48:56] = np.frombuffer(np.uint64(g.size).tobytes(), np.uint8)
        g[off_c:off_c + 4 * (nc + 1)] = np.frombuffer(offsets.astype("<u4").tobytes(), np.uint8)
        return g
    assert orc.decode(grown(offs + 1, True), 1000)[0] == oracle.ERR_CORRUPT   # offsets[0] != 0
    assert orc.decode(grown(offs, False), 1000)[0] == oracle.ERR_CORRUPT      # offsets[nc] != M
    # Chunk 2's block: its first two positions made equal, then swapped.
    # Escapes are stored one per entry in ascending order: neither is a stream.
    blk = off_d + 3 * int(offs[2])
    assert offs[3] - offs[2] >= 2
    p0, p1 = bytes(s[blk:blk + 2]), bytes(s[blk + 2:blk + 4])
    assert int.from_bytes(p0, "little") < int.from_bytes(p1, "little")
    bad = s.copy(); bad[blk + 2:blk + 4] = list(p0)
    assert orc.decode(bad, 1000)[0] == oracle.ERR_CORRUPT         # repeated position
    bad = s.copy(); bad[blk:blk + 2] = list(p1); bad[blk + 2:blk + 4] = list(p0)
    assert orc.decode(bad, 1000)[0] == oracle.ERR_CORRUPT         # falling positions
    # Damage that leaves a valid stream is accepted: a code byte changes a
    # value but breaks no rule of the format.
    off_b = 64 + pad16(1000)
    bad = s.copy(); bad[off_b + 7] ^= 0x11
    assert orc.decode(bad, 1000)[0] == oracle.OK


# ------------------------------------------------------------ plausibility

def test_gaussian_plausibility(orc):
    """Not a pin: Gaussian data with a calibrated codebook should sit in the
    page's range (Top-16 coverage above 99 %, rho just under 4/3, §3.1-§3.2)."""
    rng = np.random.default_rng(1)
    f = rng.standard_normal(1 << 20).astype(np.float32)
    x = ((f.view(np.uint32) + 0x7FFF + ((f.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    exps = orc.calibrate(x[: 1 << 16])
    rc, s = orc.encode(x, exps, 1024)
    assert rc == oracle.OK
    m = orc.count_escapes(x, exps)
    assert m / x.size < 0.01
    rho = 2 * x.size / (x.size * 1.5 + 3 * m)
    assert 1.31 < rho <= 4 / 3
