"""The PyTorch binding checks what the C ABI cannot see -- a caller-given
tensor's extent, layout and kind -- before it calls the library: a short or
strided output, a stream_bytes past the stream tensor, a short codebook, a
strided stream buffer or workspace, a status word of the wrong type, a copy
capacity past either end. Each refusal is a ValueError raised before anything
is enqueued, so the tensors around it stay untouched; the same calls with
valid arguments then succeed."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _encoded(uz, n=10_000):
    x = torch.randn(n, device="cuda").bfloat16()
    cb = uz.calibrate(x)
    stream, nbytes = uz.encode(x, cb, 1024)
    return x, cb, stream, nbytes


def test_decode_checks_its_tensors(uz):
    x, _, stream, nbytes = _encoded(uz)
    n = x.numel()
    big = torch.full((2 * n,), 7, dtype=torch.int16, device="cuda")
    bad = [
        dict(out=big[:n - 1]),  # one value short
        dict(out=big[::2]),  # strided
        dict(stream_bytes=stream.numel() + 1),  # past the stream tensor
        dict(stream_bytes=-1),
        dict(out=big[:n], status=torch.zeros(1, dtype=torch.int64, device="cuda")),
        dict(out=big[:n], status=torch.zeros(1, dtype=torch.int32)),  # pageable host memory
        dict(out=big[:n], status=torch.zeros(0, dtype=torch.int32, device="cuda")),
    ]
    for kw in bad:
        with pytest.raises(ValueError):
            uz.decode(stream, n, **kw)
    torch.cuda.synchronize()
    assert torch.all(big == 7)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    uz.decode(stream, n, out=big[:n], status=status, stream_bytes=nbytes)
    assert int(status.item()) == 0 and torch.equal(big[:n], x.view(torch.int16)) and torch.all(big[n:] == 7)


def test_e5m2_and_sentinel_decoders_check_their_outputs(uz):
    x8 = torch.randn(10_000, device="cuda").to(torch.float8_e5m2).view(torch.uint8)
    s8, n8 = uz.e5m2_encode(x8, uz.e5m2_calibrate(x8), 1024)
    with pytest.raises(ValueError):
        uz.e5m2_decode(s8, x8.numel(), out=torch.empty(x8.numel() - 1, dtype=torch.uint8, device="cuda"))
    x, cb, _, _ = _encoded(uz)
    ss, ns = uz.sentinel_encode(x, uz.make_sentinel(cb.clone()), 1024)
    with pytest.raises(ValueError):
        uz.sentinel_decode(ss, x.numel(), out=torch.empty(x.numel() - 1, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        uz.sentinel_decode(ss, x.numel(), stream_bytes=ss.numel() + 16)
    assert torch.equal(uz.e5m2_decode(s8, x8.numel(), stream_bytes=n8), x8)
    assert torch.equal(uz.sentinel_decode(ss, x.numel(), stream_bytes=ns).view(torch.int16), x.view(torch.int16))


def test_encode_checks_its_tensors(uz):
    x, cb, ref, nbytes = _encoded(uz)
    cap = ref.numel()
    with pytest.raises(ValueError):
        uz.encode(x, cb[:1024], 1024)  # short codebook
    buf = torch.full((2 * cap,), 0xAB, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        uz.encode(x, cb, 1024, out=buf[::2])  # strided stream buffer
    ws = torch.empty(2 * uz.workspace_bytes(x.numel(), 1024), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        uz.encode(x, cb, 1024, workspace=ws[::2])
    with pytest.raises(ValueError):
        uz.codebook_from_exps(list(range(16)), codebook=torch.empty(100, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(buf == 0xAB)
    # capacity is counted in bytes whatever the buffer's dtype
    out16 = torch.empty((cap + 1) // 2, dtype=torch.int16, device="cuda")
    s16, n16 = uz.encode(x, cb, 1024, out=out16)
    assert n16 == nbytes and torch.equal(s16.view(torch.uint8)[:n16], ref[:nbytes])


def test_stream_copy_and_info_check_extents(uz):
    _, _, stream, nbytes = _encoded(uz)
    dst = torch.zeros(stream.numel(), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        uz.stream_copy(stream, dst, stream.numel() + 16)
    with pytest.raises(ValueError):
        uz.stream_copy(stream, dst[: nbytes - 16], nbytes)
    with pytest.raises(ValueError):
        uz.stream_copy(stream, dst, copied=torch.zeros(1, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        uz.stream_info(stream, stream.numel() + 1)
    torch.cuda.synchronize()
    assert torch.all(dst == 0)
    copied = torch.zeros(1, dtype=torch.int64, device="cuda")
    uz.stream_copy(stream, dst, copied=copied)
    torch.cuda.synchronize()
    assert int(copied.item()) == nbytes and torch.equal(dst[:nbytes], stream[:nbytes])
    assert uz.stream_info(dst, nbytes)["total_bytes"] == nbytes
