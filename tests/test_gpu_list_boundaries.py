"""Escape counts and places that sit on the encoder's internal boundaries,
against the oracle byte for byte (SplitZip review page, §3.2: escapes are
collected per chunk in ascending position order; the stream is one fixed
layout whatever the count). The encoders keep up to 64 escapes of a
2048-value unit as a list and past that its mask bits; a warp ranks a unit's
escapes over 32 lanes of 64 positions (groups of 8 values, rows of 256).
Each unit of the input gets one pattern below: none, one at either end,
both sides of a lane's block, exactly 63 / 64 / 65 / 66 escapes packed in one
lane or spread over all, every value, group ends, a single row, random
positions; the last unit is ragged. Inputs of more than 32 units go through
the dense and escape kernels, the shorter one through the one-CTA encoder.
Integer work: the tolerance is zero."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W

pytestmark = pytest.mark.gpu

UNIT = 2048


def _patterns(rng):
    spread = lambda k: np.linspace(0, UNIT - 1, k).astype(np.int64)
    return [
        np.zeros(0, np.int64),
        np.array([0]),
        np.array([UNIT - 1]),
        np.array([63, 64]),                       # the last of lane 0's block, the first of lane 1's
        np.arange(64),                            # exactly the list's 64, all in lane 0
        np.arange(65),                            # one past it
        np.arange(64 * 5, 64 * 6),                # 64 in lane 5's block only
        np.arange(64 * 31, UNIT),                 # 64 in the last lane's block
        spread(63), spread(64), spread(65), spread(66),
        np.arange(UNIT),                          # every value
        np.arange(7, UNIT, 8)[:41],               # group ends
        np.sort(rng.choice(256, 20, replace=False)),              # the first row only
        np.sort(rng.choice(256, 20, replace=False)) + UNIT - 256,  # the last row only
        np.sort(rng.choice(UNIT, 100, replace=False)),
        np.sort(rng.choice(UNIT, 33, replace=False)),
    ]


def _layout(n, rng):
    """Escape flags of n values: unit u takes pattern u mod len(patterns);
    the ragged last unit keeps the positions below its length."""
    pats = _patterns(rng)
    esc = np.zeros(n, bool)
    for u in range((n + UNIT - 1) // UNIT):
        p = pats[u % len(pats)]
        p = p[u * UNIT + p < n]
        esc[u * UNIT + p] = True
    return esc


def _bf16(n, rng, esc):
    # codes: exponents 112..127; escapes take exponent 200 (and 0 for a few)
    e = rng.integers(112, 128, n).astype(np.uint16)
    e[esc] = np.where(rng.random(int(esc.sum())) < 0.9, 200, 0).astype(np.uint16)
    sign = rng.integers(0, 2, n).astype(np.uint16) << 15
    mant = rng.integers(0, 128, n).astype(np.uint16)
    return (sign | (e << 7) | mant).astype(np.uint16), np.arange(127, 111, -1).astype(np.uint8)


def _e5m2(n, rng, esc):
    # codes: exponents 0..15; escapes take 31 (Inf / NaN patterns) or 16..30
    e = rng.integers(0, 16, n).astype(np.uint8)
    e[esc] = np.where(rng.random(int(esc.sum())) < 0.5, 31, rng.integers(16, 31, int(esc.sum()))).astype(np.uint8)
    sign = rng.integers(0, 2, n).astype(np.uint8) << 7
    mant = rng.integers(0, 4, n).astype(np.uint8)
    return (sign | (e << 2) | mant).astype(np.uint8), np.arange(16).astype(np.uint8)


def _check(uz, orc, fmt, xh, exps, chunk):
    n = xh.size
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb = uz.codebook_from_exps([int(v) for v in exps])
    if fmt == "e5m2":
        rc, want = orc.e5m2_encode(xh, exps, chunk)
        stream, nbytes = uz.e5m2_encode(torch.from_numpy(xh).cuda(), cb, chunk)
        y = W.as_u8(uz.e5m2_decode(stream, n, stream_bytes=nbytes, status=status))
    else:
        x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
        if fmt == "sentinel":
            rc, want = orc.sentinel_encode(xh, exps, chunk)
            cb = uz.make_sentinel(cb)
            stream, nbytes = uz.sentinel_encode(x, cb, chunk)
            y = W.as_u16(uz.sentinel_decode(stream, n, stream_bytes=nbytes, status=status))
        else:
            rc, want = orc.encode(xh, exps, chunk)
            stream, nbytes = uz.encode(x, cb, chunk)
            y = W.as_u16(uz.decode(stream, n, stream_bytes=nbytes, status=status))
    assert rc == 0 and nbytes == want.size
    got = stream[:nbytes].cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"{fmt} n={n} chunk={chunk}: stream differs at {bad.size} bytes, first {bad[:8].tolist()}")
    assert int(status.item()) == 0 and np.array_equal(y, xh)


@pytest.mark.parametrize("fmt", ["bf16", "e5m2", "sentinel"])
@pytest.mark.parametrize("units", [80, 20])
@pytest.mark.parametrize("chunk", [64, 1024, 8200, 65536])
def test_escape_counts_on_the_list_and_lane_boundaries(uz, orc, fmt, units, chunk):
    rng = np.random.default_rng(units * 7 + chunk)
    n = units * UNIT + 1001
    esc = _layout(n, rng)
    xh, exps = (_e5m2 if fmt == "e5m2" else _bf16)(n, rng, esc)
    _check(uz, orc, fmt, xh, exps, chunk)
