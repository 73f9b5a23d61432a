"""The largest input the stream format holds: n = 2^32 - 1 values (chunk
offsets and escape counts are 32-bit words), for the BF16, FP8 E5M2 and
Top-15 + sentinel codecs.

The whole tensor is too large for the oracle, so each case is checked by
  - a bit-exact round trip through the GPU encoder and decoder, with guard
    words after the decoded tensor (and after the stream's capacity) that
    must stay untouched;
  - the header against the format: n, chunk, nc, M (counted here with plain
    torch ops) and the total, with offsets[0] = 0 and offsets[nc] = M;
  - slices of whole chunks -- the first ones, those across 2^31 values and
    the last ones with the ragged tail -- against the oracle's stream of the
    same values: sign-mantissa bytes, codes, offsets (rebased to the slice)
    and escape blocks.
Escapes are planted in every checked slice (a whole chunk of them near the
end, and the tensor's last values), with exponents outside the codebook.
Chunk sizes: 1024 for BF16; 8200 (not a power of two) for E5M2; 65536 for
the sentinel format, whose last chunk then spans several decoder tiles and
ends past 2^32 when its start is rounded up to whole chunks.
"""
import numpy as np
import pytest
import torch

import lossless_bf16_exponent_gb300.workloads as W
from lossless_bf16_exponent_gb300 import _lib

pytestmark = pytest.mark.gpu

N = _lib.MAX_N  # 2^32 - 1
STEP = 1 << 28  # values per generation / counting slice
GUARD = 64


def _pad16(v):
    return (v + 15) // 16 * 16


def _sections(n, chunk, fmt):
    """Section offsets of the stream format (header documentation)."""
    a_bytes = 3 * (-(-n // 8)) if fmt == "e5m2" else n
    nc = -(-n // chunk)
    off_b = 64 + _pad16(a_bytes)
    off_c = off_b + _pad16(-(-n // 2))
    off_d = off_c + _pad16(4 * (nc + 1))
    return nc, 64, off_b, off_c, off_d


def _gaussian_bits(seed, e5m2):
    """N(0, 1) bit patterns in slices (BF16 as int16, or E5M2 as uint8)."""
    out = torch.empty(N, dtype=torch.uint8 if e5m2 else torch.int16, device="cuda")
    for k, s in enumerate(range(0, N, STEP)):
        v = W.gaussian(min(STEP, N - s), seed=seed + k, device="cuda")
        out[s:s + v.numel()] = W.to_e5m2_bits(v) if e5m2 else v.view(torch.int16)
        del v
    return out


def _plant(x, chunk, patterns):
    """Escape patterns at fixed places: the first chunk, across 2^31 values,
    all of chunk nc - 3, and the tensor's last values."""
    nc = -(-N // chunk)
    pos = [0, 5, chunk - 1, (1 << 31) - 9, (1 << 31) - 1, 1 << 31, (1 << 31) + 7,
           N - 33, N - 32, N - 17, N - 9, N - 8, N - 3, N - 2, N - 1]
    idx = torch.tensor(pos, dtype=torch.int64, device="cuda")
    pat = torch.tensor([patterns[i % len(patterns)] for i in range(len(pos))], device="cuda").to(x.dtype)
    x[idx] = pat
    c = nc - 3
    full = torch.tensor(patterns, device="cuda").to(x.dtype)
    span = x[c * chunk:(c + 1) * chunk]
    span.copy_(full.repeat(-(-span.numel() // full.numel()))[:span.numel()])


def _count_escapes(x, exps, shift, mask):
    """Values whose exponent field is not one of the codebook's exponents."""
    table = torch.ones(256, dtype=torch.bool, device="cuda")
    table[torch.tensor([int(e) for e in exps], dtype=torch.int64, device="cuda")] = False
    m = 0
    for s in range(0, N, STEP):
        e = (x[s:s + STEP].to(torch.int32) >> shift) & mask
        m += int(table[e.to(torch.int64)].sum().item())
    return m


def _host(t, lo, hi):
    return t[lo:hi].cpu().numpy()


def _check_slices(stream, x, chunk, fmt, oracle_encode):
    nc, oa, ob, oc, od = _sections(N, chunk, fmt)
    esc_w = 1 if fmt == "sentinel" else 3
    starts = [0, min((1 << 31) // chunk - 2, nc // 2), nc - 4]
    for c0 in starts:
        s = c0 * chunk
        e = min(s + 4 * chunk, N)
        xs = x[s:e].cpu().numpy()
        xs = xs.view(np.uint8) if fmt == "e5m2" else xs.view(np.uint16)
        rc, want = oracle_encode(xs)
        assert rc == 0
        ns = e - s
        nc2, oa2, ob2, oc2, od2 = _sections(ns, chunk, fmt)
        a_lo, a_hi = (3 * s // 8, 3 * (-(-e // 8))) if fmt == "e5m2" else (s, e)
        assert np.array_equal(_host(stream, oa + a_lo, oa + a_hi), want[oa2:oa2 + a_hi - a_lo]), f"A at chunk {c0}"
        b_lo, b_hi = s // 2, -(-e // 2)
        assert np.array_equal(_host(stream, ob + b_lo, ob + b_hi), want[ob2:ob2 + b_hi - b_lo]), f"B at chunk {c0}"
        offs = _host(stream, oc + 4 * c0, oc + 4 * (c0 + nc2 + 1)).view(np.uint32).astype(np.int64)
        wo = want[oc2:oc2 + 4 * (nc2 + 1)].view(np.uint32).astype(np.int64)
        assert np.array_equal(offs - offs[0], wo), f"offsets at chunk {c0}"
        assert wo[-1] > 0  # planted escapes lie in every slice
        d = _host(stream, od + esc_w * int(offs[0]), od + esc_w * int(offs[-1]))
        assert np.array_equal(d, want[od2:od2 + esc_w * int(wo[-1])]), f"escapes at chunk {c0}"


def _check_header(uz, stream, nbytes, chunk, fmt, m, size_fn):
    info = uz.stream_info(stream, nbytes)
    nc, _, _, oc, _ = _sections(N, chunk, fmt)
    assert info["status"] == 0 and info["n"] == N and info["chunk"] == chunk and info["nc"] == nc
    assert info["escapes"] == m and info["total_bytes"] == nbytes == size_fn(N, m, chunk)
    assert _host(stream, oc, oc + 4).view(np.uint32)[0] == 0
    assert _host(stream, oc + 4 * nc, oc + 4 * nc + 4).view(np.uint32)[0] == m


def _decode_guarded(decode, stream, nbytes, dtype, fill):
    buf = torch.full((N + GUARD,), fill, dtype=dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    decode(stream, N, out=buf[:N], status=status, stream_bytes=nbytes)
    assert int(status.item()) == 0
    assert torch.all(buf[N:] == fill), "decoder wrote past the output"
    return buf


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _bf16_patterns(exps):
    out = [e for e in range(256) if e not in set(int(v) for v in exps)]
    pats = []
    for k, e in enumerate(out[:8]):
        pats.append(((k & 1) << 15) | (e << 7) | (k * 13 + 1) % 128)
    return [p - 65536 if p >= 32768 else p for p in pats]  # as int16


def test_bf16_max_size(uz, orc):
    chunk = 1024
    exps = orc.calibrate(W.as_u16(W.gaussian(1 << 20, seed=51)))
    cb = uz.codebook_from_exps(exps.tolist())
    x = _gaussian_bits(5100, e5m2=False)
    _plant(x, chunk, _bf16_patterns(exps))
    m = _count_escapes(x, exps, 7, 0xFF)
    cap = uz.compressed_size(N, m + 1024, chunk)
    sbuf = torch.full((cap + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    stream, nbytes = uz.encode(x.view(torch.bfloat16), cb, chunk, out=sbuf[:cap])
    assert torch.all(sbuf[cap:] == 0xA5), "encoder wrote past its capacity"
    _check_header(uz, stream, nbytes, chunk, "bf16", m, uz.compressed_size)
    _check_slices(stream, x, chunk, "bf16", lambda xs: orc.encode(xs, exps, chunk))
    buf = _decode_guarded(uz.decode, stream, nbytes, torch.int16, 0x5A5A)
    assert torch.equal(buf[:N], x)
    del x, sbuf, stream, buf
    _free()


def test_e5m2_max_size(uz, orc):
    chunk = 8200
    exps = orc.e5m2_calibrate(W.as_u8(W.to_e5m2_bits(W.gaussian(1 << 20, seed=52))))
    cb = uz.codebook_from_exps(exps.tolist())
    x = _gaussian_bits(5200, e5m2=True)
    out_e = [e for e in range(32) if e not in set(int(v) for v in exps)]
    assert out_e
    pats = [((k & 1) << 7) | (e << 2) | (k % 4) for k, e in enumerate(out_e[:8])]
    _plant(x, chunk, pats)
    m = _count_escapes(x, exps, 2, 0x1F)
    stream, nbytes = uz.e5m2_encode(x, cb, chunk, out=torch.empty(uz.e5m2_compressed_size(N, m + 1024, chunk),
                                                                  dtype=torch.uint8, device="cuda"))
    _check_header(uz, stream, nbytes, chunk, "e5m2", m, uz.e5m2_compressed_size)
    _check_slices(stream, x, chunk, "e5m2", lambda xs: orc.e5m2_encode(xs, exps, chunk))
    buf = _decode_guarded(uz.e5m2_decode, stream, nbytes, torch.uint8, 0x5A)
    assert torch.equal(buf[:N], x)
    del x, stream, buf
    _free()


def test_sentinel_max_size(uz, orc):
    chunk = 65536
    exps = orc.calibrate(W.as_u16(W.gaussian(1 << 20, seed=53)))
    cb = uz.make_sentinel(uz.codebook_from_exps(exps.tolist()))
    x = _gaussian_bits(5300, e5m2=False)
    _plant(x, chunk, _bf16_patterns(exps[:15]))
    m = _count_escapes(x, exps[:15], 7, 0xFF)  # code 15 marks every escape
    stream, nbytes = uz.sentinel_encode(x.view(torch.bfloat16), cb, chunk,
                                        out=torch.empty(uz.sentinel_compressed_size(N, m + 1024, chunk),
                                                        dtype=torch.uint8, device="cuda"))
    _check_header(uz, stream, nbytes, chunk, "sentinel", m, uz.sentinel_compressed_size)
    _check_slices(stream, x, chunk, "sentinel", lambda xs: orc.sentinel_encode(xs, exps, chunk))
    buf = _decode_guarded(uz.sentinel_decode, stream, nbytes, torch.int16, 0x5A5A)
    assert torch.equal(buf[:N], x)
    del x, stream, buf
    _free()
