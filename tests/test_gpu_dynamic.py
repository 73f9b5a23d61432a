"""GPU parity of the per-input codebook encoder (SplitZip review page, §4.3
Table 7: "dynamic Top-16"), byte for byte against the oracle.

The oracle side is the composition the page describes: the Top-16 of the
histogram of the whole input (oracle calibrate on the input itself), then the
oracle encoder with that codebook. The GPU side is one call,
uzip_encode_dynamic; its codebook tables, its stream and the decoded tensor
must all be exact.
"""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W

pytestmark = pytest.mark.gpu


def check_dynamic(uz, orc, x, chunk):
    xh = W.as_u16(x)
    exps = orc.calibrate(xh)
    rc, want = orc.encode(xh, exps, chunk)
    assert rc == 0
    stream, nbytes, cb = uz.encode_dynamic(x, chunk)
    assert uz.codebook_exps(cb) == exps.tolist()
    assert uz.codebook_histogram(cb) == [int(v) for v in orc.histogram(xh)]
    enc, dec, esc = orc.luts(exps)
    host = cb.cpu().numpy()
    assert np.array_equal(host[48:304], enc) and np.array_equal(host[32:48], dec)
    assert np.array_equal(host[304:560], esc)
    assert nbytes == want.size
    got = stream[:nbytes].cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"stream differs at {bad.size} bytes, first at {bad[:8].tolist()}")
    y = uz.decode(stream, xh.size, stream_bytes=nbytes)
    assert torch.equal(y.view(torch.int16).reshape(-1), x.reshape(-1).view(torch.int16))


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_dynamic_small(uz, orc, k):
    x, _ = W.workload(k, device="cuda", small=True)
    check_dynamic(uz, orc, x, 1024)


@pytest.mark.parametrize("chunk", [8, 256, 4096, 65536])
def test_dynamic_edge_sizes(uz, orc, chunk):
    rng = np.random.default_rng(100 + chunk)
    for n in (1, 7, 8, 9, 8191, 8192, 8193, 65537, 200_003):
        xh = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        xh[rng.random(n) < 0.05] ^= 0x3F00  # some far exponents
        x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
        check_dynamic(uz, orc, x, chunk)


def test_dynamic_empty(uz, orc):
    x = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    stream, nbytes, cb = uz.encode_dynamic(x, 1024)
    rc, want = orc.encode(np.zeros(0, np.uint16), orc.calibrate(np.zeros(0, np.uint16)), 1024)
    assert nbytes == want.size and np.array_equal(stream[:nbytes].cpu().numpy(), want)
    assert uz.codebook_exps(cb) == list(range(16))


def test_dynamic_full_kv(uz, orc):
    x, _ = W.workload(2, device="cuda")
    check_dynamic(uz, orc, x, 1024)
    del x
    torch.cuda.empty_cache()


LARGE = [(1 << 22) - 1, 1 << 22, (1 << 22) + 13, 3 * (1 << 22) + 7, 20_000_005]


@pytest.mark.parametrize("law", ["gaussian", "one exponent", "random bits"])
def test_histogram_of_large_inputs(uz, orc, law):
    """Inputs of 4 Mi values and more are counted by the private-column
    histogram (one CTA per SM, 16-bit counters per thread): histogram and
    codebook equal the oracle's, at and around the size where it takes over,
    with ragged tails and inputs spanning several rounds of loads."""
    rng = np.random.default_rng(len(law))
    for n in LARGE:
        if law == "gaussian":
            xh = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        elif law == "one exponent":  # every pair of counts hits one counter
            xh = np.full(n, 0x3F85, np.uint16)
            xh[::1001] = 0x4005
        else:
            xh = rng.integers(0, 65536, n, dtype=np.uint16)
        x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
        cb = uz.calibrate(x)
        assert uz.codebook_histogram(cb) == [int(v) for v in orc.histogram(xh)], n
        assert uz.codebook_exps(cb) == orc.calibrate(xh).tolist(), n


def test_e5m2_histogram_of_large_inputs(uz, orc):
    rng = np.random.default_rng(9)
    for n in LARGE:
        xh = rng.integers(0, 256, n, dtype=np.uint8)
        xh[: n // 3] = 0x3C  # a dominant exponent
        cb = uz.e5m2_calibrate(torch.from_numpy(xh).cuda())
        assert uz.codebook_histogram(cb) == [int(v) for v in orc.e5m2_histogram(xh)], n
        assert uz.codebook_exps(cb) == orc.e5m2_calibrate(xh).tolist(), n
