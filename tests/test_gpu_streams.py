"""Concurrent use: the entry points that take the caller's buffers keep no
device state between calls, so calls on different CUDA streams, each with its
own output, workspace and codebook, may run at the same time on the GPU.
(uzip_encode_noalloc is the exception: every call shares one built-in scratch
array, so its calls must be serialised; it is not used here.) Two tensors are encoded and decoded on
two streams at once; each stream must equal, byte for byte, the stream the
same call produces alone on the default stream, and each round trip must be
bit-exact."""
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W

pytestmark = pytest.mark.gpu


# 4 Mi values each: the two-kernel path, enough blocks for the two to overlap;
# 150,000 each: one thread-block cluster each, side by side
@pytest.mark.parametrize("values", [1 << 22, 150_000])
def test_two_streams_at_once_match_sequential_calls(uz, values):
    dev = torch.device("cuda")
    shape = (values // (2 * 8 * 256 * 128) or 1, 2, 8, 256, 128)
    kv = W.kv_cache(shape, seed=21, device=dev).reshape(-1)[:values]
    xs = [kv.contiguous(), W.heavy_tailed(values, seed=22, device=dev)]
    samples = [W.kv_cache_sample(device=dev), W.gaussian(1 << 16, seed=23, device=dev)]
    chunks = [1024, 256]
    cbs = [uz.calibrate(s) for s in samples]
    want = [uz.encode(x, cb, c) for x, cb, c in zip(xs, cbs, chunks)]
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream(dev) for _ in xs]
    outs = [torch.empty(uz.max_compressed_size(x.numel(), c), dtype=torch.uint8, device=dev)
            for x, c in zip(xs, chunks)]
    wss = [torch.empty(uz.workspace_bytes(x.numel(), c), dtype=torch.uint8, device=dev) for x, c in zip(xs, chunks)]
    ys = [torch.empty_like(x) for x in xs]
    for rep in range(3):
        for o in outs:
            o.fill_(0xAB)
        torch.cuda.synchronize()
        for k, st in enumerate(streams):
            with torch.cuda.stream(st):
                uz.encode(xs[k], cbs[k], chunks[k], out=outs[k], workspace=wss[k], sync=False)
                uz.decode(outs[k], xs[k].numel(), out=ys[k])
        torch.cuda.synchronize()
        for k in range(len(xs)):
            stream, nbytes = want[k]
            assert torch.equal(outs[k][:nbytes], stream[:nbytes]), f"stream {k} differs (rep {rep})"
            assert torch.all(outs[k][nbytes:] == 0xAB), f"stream {k}: bytes past its end written (rep {rep})"
            assert torch.equal(ys[k].view(torch.int16), xs[k].view(torch.int16)), f"round trip {k} (rep {rep})"
