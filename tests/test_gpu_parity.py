"""GPU parity: the sm_103a kernels against the CPU oracle, byte for byte.

For every case the same seeded input goes to both sides:
  - calibration: histogram, Top-16 codebook and all three tables equal;
  - encode: the GPU stream equals the oracle stream byte for byte (header,
    sections, padding, escape blocks);
  - decode: the GPU decoder rebuilds the input bit-exactly from the GPU stream
    and from the oracle's stream.
Codec work is integer and byte work, so the bar is exact equality throughout.
Cases: oracle-sized instances of every workload law spanning many tiles with a
ragged tail, edge sizes around tile and chunk boundaries for many chunk sizes,
degenerate inputs, and the full-size workloads the benchmark runs.
"""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W

pytestmark = pytest.mark.gpu


def u16(x):
    return W.as_u16(x)


def check_codebook(uz, orc, cb, sample_u16):
    """The GPU codebook against the oracle's; returns the oracle's exponents
    (the oracle's inputs never come from the CUDA path)."""
    exps = orc.calibrate(sample_u16)
    assert uz.codebook_exps(cb) == exps.tolist()
    assert uz.codebook_histogram(cb) == [int(v) for v in orc.histogram(sample_u16)]
    enc, dec, esc = orc.luts(exps)
    host = cb.cpu().numpy()
    assert np.array_equal(host[48:304], enc)
    assert np.array_equal(host[32:48], dec)
    assert np.array_equal(host[304:560], esc)
    return exps


def check_codec(uz, orc, x, exps, cb, chunk):
    """Encode on both sides, compare streams, decode both streams on the GPU."""
    xh = u16(x)
    n = xh.size
    rc, want = orc.encode(xh, exps, chunk)
    assert rc == 0
    stream, nbytes = uz.encode(x, cb, chunk)
    assert nbytes == want.size
    got = stream[:nbytes].cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"stream differs at {bad.size} bytes, first at {bad[:8].tolist()} of {nbytes}")
    status = torch.zeros(1, dtype=torch.int32, device=x.device)
    y = uz.decode(stream, n, stream_bytes=nbytes, status=status)
    assert int(status.item()) == 0
    assert torch.equal(y.view(torch.int16).reshape(-1), x.reshape(-1).view(torch.int16))
    y2 = uz.decode(torch.from_numpy(want).to(x.device), n, status=status)
    assert int(status.item()) == 0
    assert torch.equal(y2.view(torch.int16).reshape(-1), x.reshape(-1).view(torch.int16))
    info = uz.stream_info(stream, nbytes)
    assert info["status"] == 0 and info["total_bytes"] == nbytes
    return int(info["escapes"])


# ------------------------------------------------------ oracle-sized workloads

@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_workload_small(uz, orc, k):
    x, s = W.workload(k, device="cuda", small=True)
    cb = uz.calibrate(s)
    exps = check_codebook(uz, orc, cb, u16(s))
    check_codec(uz, orc, x, exps, cb, 1024)


@pytest.mark.parametrize("chunk", W.SWEEP_CHUNKS)
def test_sweep_small(uz, orc, chunk):
    s = W.sweep_sample("cuda", n=1 << 16)
    cb = uz.calibrate(s)
    exps = check_codebook(uz, orc, cb, u16(s))
    for nbytes in W.SWEEP_BYTES[:8]:  # 4 KiB .. 512 KiB
        check_codec(uz, orc, W.sweep(nbytes, "cuda"), exps, cb, chunk)


# ----------------------------------------------------------------- edge sizes

EDGE_CHUNKS = [8, 24, 256, 512, 1000, 1024, 2048, 4096, 8192, 8200, 16384, 32768, 63496, 64008, 65528, 65536]


@pytest.mark.parametrize("chunk", EDGE_CHUNKS)
def test_edge_sizes(uz, orc, chunk):
    rng = np.random.default_rng(chunk)
    sizes = sorted({1, 2, 7, 8, 9, 15, 17, chunk - 1, chunk, chunk + 1, 3 * chunk + 5, 8191, 8192, 8193,
                    2 * 8192 + 9, 65537, 200_003})
    for n in sizes:
        if rng.random() < 0.5:  # random bit patterns: about 94 % escapes
            xh = rng.integers(0, 65536, n).astype(np.uint16)
        else:  # Gaussian bits: few escapes
            xh = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
        exps = rng.choice(256, 16, replace=False).astype(np.uint8)
        if rng.random() < 0.5:
            exps = orc.calibrate(xh)
        cb = uz.codebook_from_exps(exps.tolist())
        check_codec(uz, orc, x, exps, cb, chunk)


def test_empty_input(uz, orc):
    exps = np.arange(16, dtype=np.uint8)
    cb = uz.codebook_from_exps(exps.tolist())
    x = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    for chunk in (8, 1024, 65536):
        rc, want = orc.encode(np.zeros(0, np.uint16), exps, chunk)
        stream, nbytes = uz.encode(x, cb, chunk)
        assert nbytes == want.size == 80
        assert np.array_equal(stream[:nbytes].cpu().numpy(), want)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        uz.decode(stream, 0, stream_bytes=nbytes, status=status)
        assert int(status.item()) == 0


@pytest.mark.parametrize("chunk", [8, 256, 512, 1024, 2048, 4096, 65536])
def test_degenerate_inputs(uz, orc, chunk):
    n = 3 * 65536 + 11
    cases = {
        "all zero": np.zeros(n, np.uint16),
        "all escape": np.full(n, 0x3F80, np.uint16),  # exponent 0x7F, not in codes 0..15
        "all patterns": np.tile(np.arange(65536, dtype=np.uint32).astype(np.uint16), 3)[:n],
        "specials": np.tile(np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F],
                                     np.uint16), n // 8 + 1)[:n],
    }
    for name, xh in cases.items():
        x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
        for exps in (np.arange(16, dtype=np.uint8), orc.calibrate(xh)):
            cb = uz.codebook_from_exps(exps.tolist())
            m = check_codec(uz, orc, x, exps, cb, chunk)
            if name == "all escape" and exps[0] == 0:
                assert m == n


def test_calibration_edge_samples(uz, orc):
    rng = np.random.default_rng(4)
    for n in (0, 1, 7, 8, 9, 1000, (1 << 16) + 3):
        xh = rng.integers(0, 65536, n).astype(np.uint16)
        xh[: n // 2] = 0x3F80  # a dominant exponent
        x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
        cb = uz.calibrate(x)
        check_codebook(uz, orc, cb, xh)


# ------------------------------------------------------------ full workloads

@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_workload_full(uz, orc, k):
    x, s = W.workload(k, device="cuda")
    cb = uz.calibrate(s)
    exps = check_codebook(uz, orc, cb, u16(s))
    m = check_codec(uz, orc, x, exps, cb, 1024)
    eps = m / x.numel()
    if k == 2:
        assert eps < 0.01  # KV-shaped: the page's regime (>99 % coverage)
    if k == 3:
        assert 0.01 < eps < 0.08  # escape stress: a few percent
    del x, s
    torch.cuda.empty_cache()


@pytest.mark.parametrize("chunk", W.SWEEP_CHUNKS)
def test_sweep_full(uz, orc, chunk):
    s = W.sweep_sample("cuda")
    cb = uz.calibrate(s)
    exps = check_codebook(uz, orc, cb, u16(s))
    for nbytes in W.SWEEP_BYTES:
        check_codec(uz, orc, W.sweep(nbytes, "cuda"), exps, cb, chunk)
    torch.cuda.empty_cache()
