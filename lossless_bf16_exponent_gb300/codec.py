"""PyTorch front end of libuzip: device buffers and the current CUDA stream
go in, the C ABI does all the work. Tensors must be contiguous CUDA tensors
with 16-byte aligned storage; BF16 data may be any 2-byte dtype (the codec
works on bit patterns)."""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import CODEBOOK_BYTES, HEADER_BYTES, UzipError, check


# The current stream's raw handle without building a Stream object (a few
# microseconds per call otherwise); the public API where this is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _sp(device=None) -> int:
    """Raw handle of the current CUDA stream of ``device`` (default: current device)."""
    if _raw_stream is not None:
        if isinstance(device, torch.device):
            idx = device.index
        else:
            idx = device
        return _raw_stream(torch.cuda.current_device() if idx is None else idx)
    return torch.cuda.current_stream(device).cuda_stream


def _p(t: torch.Tensor | None):
    return t.data_ptr() if t is not None else None


def _flat16(x: torch.Tensor) -> torch.Tensor:
    """Check a tensor of 16-bit values for the C ABI (CUDA, contiguous); the
    tensor itself is returned (the ABI takes its pointer and element count)."""
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if x.element_size() != 2:
        raise ValueError(f"expected 16-bit values, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _dev(t: torch.Tensor, what: str, nbytes: int = 0) -> torch.Tensor:
    """Check a caller-given device buffer: a contiguous CUDA tensor of at
    least ``nbytes`` bytes (the C ABI takes only its address, so its extent
    is checked here)."""
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    if _nbytes(t) < nbytes:
        raise ValueError(f"{what}: holds {_nbytes(t)} bytes, needs {nbytes}")
    return t


def _cb(codebook: torch.Tensor) -> torch.Tensor:
    return _dev(codebook, "codebook", CODEBOOK_BYTES)


def _status(status: torch.Tensor | None):
    """The decoders' status word: one int32 in device (or pinned host) memory."""
    if status is None:
        return None
    if (status.dtype != torch.int32 or status.numel() < 1 or not status.is_contiguous()
            or not (status.is_cuda or status.is_pinned())):
        raise ValueError("status: expected a contiguous int32 CUDA (or pinned host) tensor of one element")
    return _p(status)


def _stream_nbytes(stream: torch.Tensor, stream_bytes: int | None) -> int:
    """Readable bytes of a stream tensor: all of it, or the first ``stream_bytes``."""
    if not stream.is_contiguous():
        raise ValueError("stream: expected a contiguous tensor")
    if stream_bytes is None:
        return _nbytes(stream)
    if not 0 <= stream_bytes <= _nbytes(stream):
        raise ValueError(f"stream_bytes {stream_bytes} outside the stream tensor ({_nbytes(stream)} bytes)")
    return int(stream_bytes)


def _out_values(out: torch.Tensor, n: int, flat) -> torch.Tensor:
    """A caller-given output of n values (``flat`` checks the element size)."""
    o = flat(out)
    if o.numel() < n:
        raise ValueError(f"out: holds {o.numel()} values, needs {n}")
    return o


def load():
    return _lib.load()


# ---------------------------------------------------------------- codebook

def new_codebook(device="cuda") -> torch.Tensor:
    return torch.empty(CODEBOOK_BYTES, dtype=torch.uint8, device=device)


def calibrate(sample: torch.Tensor, codebook: torch.Tensor | None = None) -> torch.Tensor:
    """Top-16 codebook from the exponent histogram of ``sample`` (offline
    calibration, SplitZip §3.3). Returns the 4096-byte device codebook."""
    s = _flat16(sample)
    cb = new_codebook(s.device) if codebook is None else _cb(codebook)
    check(load().uzip_calibrate(_p(s), s.numel(), _p(cb), _sp(s.device)), "uzip_calibrate")
    return cb


def codebook_from_exps(exps, device="cuda", codebook: torch.Tensor | None = None) -> torch.Tensor:
    vals = [int(v) for v in exps]
    if len(vals) != 16:
        raise ValueError("need 16 exponents")
    arr = (ctypes.c_uint8 * 16)(*vals)
    cb = new_codebook(device) if codebook is None else _cb(codebook)
    check(load().uzip_codebook_from_exps(arr, _p(cb), _sp(cb.device)), "uzip_codebook_from_exps")
    return cb


def codebook_exps(codebook: torch.Tensor) -> list[int]:
    """The 16 exponents of a codebook (copies to the host)."""
    return codebook[_lib.CB_EXPS:_lib.CB_EXPS + 16].cpu().tolist()


def codebook_histogram(codebook: torch.Tensor) -> list[int]:
    h = codebook[_lib.CB_HIST:_lib.CB_HIST + 2048].cpu().view(torch.int64)
    return [int(v) for v in h.tolist()]


# ------------------------------------------------------------------- sizes

def compressed_size(n: int, n_escapes: int, chunk: int = 1024) -> int:
    return int(load().uzip_compressed_size(n, n_escapes, chunk))


def max_compressed_size(n: int, chunk: int = 1024) -> int:
    return compressed_size(n, n, chunk)


def workspace_bytes(n: int, chunk: int = 1024) -> int:
    return int(load().uzip_encode_workspace_bytes(n, chunk))


# ------------------------------------------------------------------ codec

def encode(x: torch.Tensor, codebook: torch.Tensor, chunk: int = 1024, out: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None, sync: bool = True):
    """Encode ``x`` (SplitZip §3.2). Returns ``(stream, nbytes)``; ``stream``
    is the whole output buffer, ``nbytes`` the exact stream size (None when
    ``sync=False``: read it later with :func:`stream_info`)."""
    v = _flat16(x)
    n = v.numel()
    if out is None:
        out = torch.empty(max_compressed_size(n, chunk), dtype=torch.uint8, device=v.device)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_bytes(n, chunk)), dtype=torch.uint8, device=v.device)
    nbytes = ctypes.c_size_t(0)
    L = load()
    args = (_p(v), n, chunk, _p(_cb(codebook)), _p(_dev(out, "out")), _nbytes(out),
            _p(_dev(workspace, "workspace")), _nbytes(workspace), ctypes.byref(nbytes) if sync else None)
    check(L.uzip_encode(*args, _sp(v.device)), "uzip_encode")
    return out, (nbytes.value if sync else None)


def encode_dynamic(x: torch.Tensor, chunk: int = 1024, codebook: torch.Tensor | None = None,
                   out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, sync: bool = True):
    """Encode ``x`` with a codebook built from ``x`` itself (SplitZip §4.3,
    Table 7). Returns ``(stream, nbytes, codebook)``."""
    v = _flat16(x)
    n = v.numel()
    cb = new_codebook(v.device) if codebook is None else _cb(codebook)
    if out is None:
        out = torch.empty(max_compressed_size(n, chunk), dtype=torch.uint8, device=v.device)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_bytes(n, chunk)), dtype=torch.uint8, device=v.device)
    nbytes = ctypes.c_size_t(0)
    args = (_p(v), n, chunk, _p(cb), _p(_dev(out, "out")), _nbytes(out), _p(_dev(workspace, "workspace")),
            _nbytes(workspace), ctypes.byref(nbytes) if sync else None)
    check(load().uzip_encode_dynamic(*args, _sp(v.device)), "uzip_encode_dynamic")
    return out, (nbytes.value if sync else None), cb


def decode(stream: torch.Tensor, n: int, out: torch.Tensor | None = None, status: torch.Tensor | None = None,
           stream_bytes: int | None = None, dtype=torch.bfloat16) -> torch.Tensor:
    """Decode ``n`` values from a stream (SplitZip §3.2). Device-side errors
    land in ``status`` (a 1-element int32 CUDA tensor) when given."""
    if out is None:
        out = torch.empty(n, dtype=dtype, device=stream.device)
    o = _out_values(out, n, _flat16) if n else out
    nb = _stream_nbytes(stream, stream_bytes)
    check(load().uzip_decode(_p(stream), nb, _p(o) if n else None, n, _status(status), _sp(stream.device)),
          "uzip_decode")
    return out


def stream_copy(src: torch.Tensor, dst: torch.Tensor, capacity: int | None = None,
                copied: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> None:
    """Copy the stream at ``src`` (exactly its header's total bytes) to
    ``dst``; either may be pinned host memory. ``copied`` (one int64 element,
    device or pinned host) receives the byte count. Asynchronous on ``stream``
    (default: the current stream of the device)."""
    for t, what in ((src, "src"), (dst, "dst")):
        if not t.is_contiguous():
            raise ValueError(f"{what}: expected a contiguous tensor")
    room = min(_nbytes(src), _nbytes(dst))
    cap = room if capacity is None else int(capacity)
    if not 0 <= cap <= room:
        raise ValueError(f"capacity {cap} beyond src or dst ({room} bytes)")
    if copied is not None and (copied.dtype != torch.int64 or copied.numel() < 1 or not copied.is_contiguous()):
        raise ValueError("copied: expected a contiguous int64 tensor of one element")
    dev = src.device if src.is_cuda else dst.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    check(load().uzip_stream_copy(_p(src), _p(dst), cap, _p(copied), ctypes.c_void_p(s.cuda_stream)),
          "uzip_stream_copy")


def stream_info(stream: torch.Tensor, stream_bytes: int | None = None) -> dict:
    info = _lib.Info()
    nb = _stream_nbytes(stream, stream_bytes)
    rc = load().uzip_stream_info(_p(stream), nb, ctypes.byref(info), _sp(stream.device))
    d = {f: getattr(info, f) for f, _ in _lib.Info._fields_ if f != "exps"}
    d["exps"] = list(info.exps)
    d["status"] = rc
    return d


def roundtrip_ok(x: torch.Tensor, codebook: torch.Tensor, chunk: int = 1024) -> bool:
    s, nb = encode(x, codebook, chunk)
    y = decode(s, x.numel(), stream_bytes=nb, dtype=x.dtype)
    return bool(torch.equal(y.view(torch.int16), _flat16(x).reshape(-1).view(torch.int16)))


__all__ = [
    "HEADER_BYTES", "CODEBOOK_BYTES", "UzipError", "load", "new_codebook", "calibrate", "codebook_from_exps",
    "codebook_exps", "codebook_histogram", "compressed_size", "max_compressed_size", "workspace_bytes",
    "encode", "decode", "stream_info", "roundtrip_ok",
]


# ------------------------------------------------------------ FP8 E5M2

def _flat8(x: torch.Tensor) -> torch.Tensor:
    if not x.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if x.element_size() != 1:
        raise TypeError("expected one-byte FP8 E5M2 values (torch.float8_e5m2 or uint8 bit patterns)")
    if not x.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return x.reshape(-1).view(torch.uint8)


def e5m2_calibrate(sample: torch.Tensor, codebook: torch.Tensor | None = None) -> torch.Tensor:
    """Codebook from E5M2 values (SplitZip §4.2 / appendix C)."""
    s = _flat8(sample)
    cb = new_codebook(s.device) if codebook is None else _cb(codebook)
    check(load().uzip_e5m2_calibrate(_p(s), s.numel(), _p(cb), _sp(s.device)), "uzip_e5m2_calibrate")
    return cb


def e5m2_compressed_size(n: int, n_escapes: int, chunk: int = 1024) -> int:
    return int(load().uzip_e5m2_compressed_size(n, n_escapes, chunk))


def e5m2_encode(x: torch.Tensor, codebook: torch.Tensor, chunk: int = 1024, out: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, sync: bool = True):
    """Encode E5M2 values; returns ``(stream, nbytes)`` as :func:`encode`."""
    v = _flat8(x)
    n = v.numel()
    if out is None:
        out = torch.empty(e5m2_compressed_size(n, n, chunk), dtype=torch.uint8, device=v.device)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_bytes(n, chunk)), dtype=torch.uint8, device=v.device)
    nbytes = ctypes.c_size_t(0)
    args = (_p(v), n, chunk, _p(_cb(codebook)), _p(_dev(out, "out")), _nbytes(out),
            _p(_dev(workspace, "workspace")), _nbytes(workspace), ctypes.byref(nbytes) if sync else None)
    check(load().uzip_e5m2_encode(*args, _sp(v.device)), "uzip_e5m2_encode")
    return out, (nbytes.value if sync else None)


def e5m2_decode(stream: torch.Tensor, n: int, out: torch.Tensor | None = None, status: torch.Tensor | None = None,
                stream_bytes: int | None = None) -> torch.Tensor:
    """Decode an E5M2 stream into ``n`` bytes (uint8 bit patterns)."""
    if out is None:
        out = torch.empty(max(n, 1), dtype=torch.uint8, device=stream.device)[:n]
    o = _out_values(out, n, _flat8) if n else out
    nb = _stream_nbytes(stream, stream_bytes)
    check(load().uzip_e5m2_decode(_p(stream), nb, _p(o) if n else None, n, _status(status), _sp(stream.device)),
          "uzip_e5m2_decode")
    return out


# ------------------------------------------------------ Top-15 + sentinel

def make_sentinel(codebook: torch.Tensor) -> torch.Tensor:
    """Turn a codebook into the Top-15 + sentinel codebook of its first 15
    exponents, in place (SplitZip §3.4, Table 6)."""
    check(load().uzip_codebook_make_sentinel(_p(_cb(codebook)), _sp(codebook.device)), "uzip_codebook_make_sentinel")
    return codebook


def sentinel_compressed_size(n: int, n_escapes: int, chunk: int = 1024) -> int:
    return int(load().uzip_sentinel_compressed_size(n, n_escapes, chunk))


def sentinel_encode(x: torch.Tensor, codebook: torch.Tensor, chunk: int = 1024, out: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, sync: bool = True):
    """Encode BF16 values in the Top-15 + sentinel format; ``(stream, nbytes)``."""
    v = _flat16(x)
    n = v.numel()
    if out is None:
        out = torch.empty(sentinel_compressed_size(n, n, chunk), dtype=torch.uint8, device=v.device)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_bytes(n, chunk)), dtype=torch.uint8, device=v.device)
    nbytes = ctypes.c_size_t(0)
    args = (_p(v), n, chunk, _p(_cb(codebook)), _p(_dev(out, "out")), _nbytes(out),
            _p(_dev(workspace, "workspace")), _nbytes(workspace), ctypes.byref(nbytes) if sync else None)
    check(load().uzip_sentinel_encode(*args, _sp(v.device)), "uzip_sentinel_encode")
    return out, (nbytes.value if sync else None)


def sentinel_decode(stream: torch.Tensor, n: int, out: torch.Tensor | None = None,
                    status: torch.Tensor | None = None, stream_bytes: int | None = None) -> torch.Tensor:
    """Decode a Top-15 + sentinel stream into ``n`` BF16 values."""
    if out is None:
        out = torch.empty(max(n, 1), dtype=torch.bfloat16, device=stream.device)[:n]
    o = _out_values(out, n, _flat16) if n else out
    nb = _stream_nbytes(stream, stream_bytes)
    check(load().uzip_sentinel_decode(_p(stream), nb, _p(o) if n else None, n, _status(status),
                                      _sp(stream.device)),
          "uzip_sentinel_decode")
    return out
