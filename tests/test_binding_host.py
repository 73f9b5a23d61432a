"""The binding's own checks that need no GPU: readable stream extents, the
status word's type and memory, and a copy's capacity against both ends, all
refused with ValueError before the library is called."""
import pytest
import torch

from lossless_bf16_exponent_gb300 import codec


def test_stream_extent():
    s = torch.zeros(100, dtype=torch.uint8)
    assert codec._stream_nbytes(s, None) == 100
    assert codec._stream_nbytes(s, 64) == 64
    assert codec._stream_nbytes(torch.zeros(10, dtype=torch.int32), None) == 40  # counted in bytes
    for bad in (101, -1):
        with pytest.raises(ValueError):
            codec._stream_nbytes(s, bad)
    with pytest.raises(ValueError):
        codec._stream_nbytes(torch.zeros(200, dtype=torch.uint8)[::2], None)


def test_status_word():
    assert codec._status(None) is None
    for bad in (torch.zeros(1, dtype=torch.int32),  # pageable host memory
                torch.zeros(1, dtype=torch.int64),
                torch.zeros(0, dtype=torch.int32)):
        with pytest.raises(ValueError):
            codec._status(bad)


def test_device_buffers_and_codebook():
    with pytest.raises(ValueError):
        codec._dev(torch.zeros(16, dtype=torch.uint8), "out")  # not on the device
    with pytest.raises(ValueError):
        codec._cb(torch.zeros(4096, dtype=torch.uint8))
    with pytest.raises(ValueError):
        codec._flat16(torch.zeros(4, dtype=torch.int16))


def test_stream_copy_capacity_within_both_ends():
    src = torch.zeros(256, dtype=torch.uint8)
    dst = torch.zeros(128, dtype=torch.uint8)
    with pytest.raises(ValueError, match="capacity"):
        codec.stream_copy(src, dst, 129)
    with pytest.raises(ValueError, match="capacity"):
        codec.stream_copy(src, dst, -1)
    with pytest.raises(ValueError, match="contiguous"):
        codec.stream_copy(src[::2], dst, 64)
    with pytest.raises(ValueError, match="copied"):
        codec.stream_copy(src, dst, 64, copied=torch.zeros(1, dtype=torch.int32))
    assert torch.all(dst == 0)
