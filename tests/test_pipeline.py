"""Streamed transfer in compressed form (SplitZip review page, appendix B):
piece splitting and the stage model on the CPU; the GPU pipeline's output
bit-identical to its input, each piece's bytes equal to the oracle's stream
of that piece."""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib
from lossless_bf16_exponent_gb300 import pipeline as PL


@pytest.mark.parametrize("n,pieces", [(1, 1), (7, 3), (8, 2), (1000, 7), (8192, 16), (100_003, 5), (64, 64)])
def test_split_points_cover_and_align(n, pieces):
    parts = PL.split_points(n, pieces)
    assert parts[0][0] == 0 and parts[-1][1] == n
    assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
    assert all(s % 8 == 0 and e > s for s, e in parts)
    assert len(parts) <= pieces


def test_split_points_degenerate():
    assert PL.split_points(0, 4) == [] and PL.split_points(10, 0) == []


def test_b_hide_and_model():
    # the page's own numbers: 613.3 GB/s encode, 2181.8 decode, ratio 1.324 -> about 463.2 GB/s
    assert abs(PL.b_hide(613.3, 2181.8, 1.324) - 463.2) < 0.1
    # a link slower than B_hide: the transfer stage sets the pace
    t = PL.model_seconds(10**9, 600e9, 2000e9, 1.3, 100e9, pieces=10**6)
    assert abs(t - 10**9 / (1.3 * 100e9)) < 1e-6
    # a link faster than B_hide: the encoder sets the pace
    t = PL.model_seconds(10**9, 600e9, 2000e9, 1.3, 10**13, pieces=10**6)
    assert abs(t - 10**9 / 600e9) < 1e-6


@pytest.mark.gpu
@pytest.mark.parametrize("link", ["host", "d2d"])
def test_pipeline_round_trip_and_piece_streams(uz, orc, link):
    x, s = W.workload(1, device="cuda")  # 1,048,576 values
    cb = uz.calibrate(s)
    exps = orc.calibrate(W.as_u16(s))
    assert uz.codebook_exps(cb) == exps.tolist()
    y, tr = PL.send_compressed(x, cb, chunk=1024, pieces=6, link=link)
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))
    xh = W.as_u16(x)
    want = sum(orc.encode(xh[a:b], exps, 1024)[1].size for a, b in PL.split_points(xh.size, 6))
    assert tr.sent_bytes == want and tr.pieces == 6
    yr, trr = PL.send_raw(x, pieces=6, link=link)
    assert torch.equal(yr.view(torch.int16), x.view(torch.int16)) and trr.sent_bytes == 2 * xh.size


@pytest.mark.gpu
def test_pipeline_odd_sizes(uz, orc):
    rng = np.random.default_rng(9)
    xh = (rng.standard_normal(200_003).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
    cb = uz.calibrate(x[:65536])
    for pieces in (1, 3, 40):
        y, _ = PL.send_compressed(x, cb, chunk=256, pieces=pieces, link="host")
        assert torch.equal(y.view(torch.int16), x.view(torch.int16))


@pytest.mark.gpu
def test_stream_copy_exact_bytes(uz, orc):
    x, s = W.workload(1, device="cuda")
    cb = uz.calibrate(s)
    stream, nbytes = uz.encode(x, cb, 1024)
    cap = stream.numel()
    copied = torch.zeros(1, dtype=torch.int64, device="cuda")
    for dst in (torch.full((cap,), 0xAB, dtype=torch.uint8, device="cuda"),
                torch.full((cap,), 0xAB, dtype=torch.uint8).pin_memory()):
        uz.stream_copy(stream, dst, cap, copied=copied)
        torch.cuda.synchronize()
        assert int(copied.item()) == nbytes
        d = dst.cpu()
        assert torch.equal(d[:nbytes], stream[:nbytes].cpu()) and torch.all(d[nbytes:] == 0xAB)
        back = torch.full((cap,), 0xCD, dtype=torch.uint8, device="cuda")
        uz.stream_copy(dst, back, cap, copied=copied)  # host (or device) -> device
        torch.cuda.synchronize()
        assert int(copied.item()) == nbytes and torch.equal(back[:nbytes], stream[:nbytes])
        assert torch.all(back[nbytes:] == 0xCD)


@pytest.mark.gpu
def test_stream_copy_refuses_non_streams(uz):
    junk = torch.randint(0, 255, (4096,), dtype=torch.uint8, device="cuda")
    dst = torch.full((4096,), 7, dtype=torch.uint8, device="cuda")
    copied = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    uz.stream_copy(junk, dst, 4096, copied=copied)
    torch.cuda.synchronize()
    assert int(copied.item()) == 0 and torch.all(dst == 7)
    x = torch.randn(10_000, device="cuda").bfloat16()
    stream, nbytes = uz.encode(x, uz.calibrate(x), 1024)
    dst = torch.full((stream.numel(),), 7, dtype=torch.uint8, device="cuda")
    uz.stream_copy(stream, dst, nbytes - 1, copied=copied)  # capacity below the stream's total
    torch.cuda.synchronize()
    assert int(copied.item()) == 0 and torch.all(dst == 7)


@pytest.mark.gpu
def test_stream_copy_refuses_pageable_memory(uz):
    """A kernel may touch device or pinned host memory only: pageable host
    buffers (either end, or the byte-count word) are refused on the host,
    before anything is launched."""
    x = torch.randn(10_000, device="cuda").bfloat16()
    stream, nbytes = uz.encode(x, uz.calibrate(x), 1024)
    cap = stream.numel()
    dst = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(cap, dtype=torch.uint8)
    assert not pageable.is_pinned()
    for src, to in ((stream, pageable), (pageable, dst)):
        with pytest.raises(_lib.UzipError) as e:
            uz.stream_copy(src, to, cap)
        assert e.value.code == _lib.ERR_ARG
    with pytest.raises(_lib.UzipError) as e:
        uz.stream_copy(stream, dst, cap, copied=torch.zeros(1, dtype=torch.int64))
    assert e.value.code == _lib.ERR_ARG
    torch.cuda.synchronize()
    assert torch.all(dst == 0) and torch.all(pageable == 0)
