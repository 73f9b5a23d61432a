"""Streamed transfer of a BF16 tensor in compressed form: encode -> link -> decode.

SplitZip review page, §4.4 / appendix B: compression, transfer and
decompression form a streaming pipeline. With raw size S, ratio rho, encode
and decode throughputs G_enc and G_dec and link bandwidth B, the stages take
T_enc = S / G_enc, T_xfer = S / (rho B) and T_dec = S / G_dec; the steady
state runs at the slowest stage, and the codec is fully hidden for any link
up to B_hide = min(G_enc, G_dec) / rho.

Here the tensor is cut into pieces that each become their own stream. Piece
k is encoded on one CUDA stream, sent over the link on a second (and, for the
host link, received on a third), and decoded on a fourth, each stage waiting
only for the previous stage of the same piece, so piece k+1 is encoded while
piece k travels. Two links stand in for the network on one GPU:

  "host"  device -> pinned host memory -> device (the NVLink-C2C link of a
          Grace-Blackwell node, both directions busy at once);
  "d2d"   a device-to-device copy inside HBM.

A piece's compressed length is known only on the device (in its stream
header). On the d2d link each hop is a uzip_stream_copy, which reads the
length there, so the host enqueues every stage up front and never waits. The
host link uses the copy engines (copy kernels would wait for SMs that the
codec kernels occupy), which need the length on the host: the sender reads
piece k's 64-byte header while piece k + 1 is already encoding, well within
the time the link takes per piece.

Everything on the data path runs in libuzip's kernels and CUDA copies; this
module only orders them.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from .codec import _flat16, _p, check, load, max_compressed_size, stream_copy, workspace_bytes


def split_points(n: int, pieces: int) -> list[tuple[int, int]]:
    """[start, end) of each piece: near-equal sizes, every start a multiple of
    8 values (16-byte aligned, as the codec requires); empty pieces dropped."""
    if n <= 0 or pieces <= 0:
        return []
    per = -(-n // pieces)
    per = -(-per // 8) * 8
    out = []
    s = 0
    while s < n:
        e = min(n, s + per)
        out.append((s, e))
        s = e
    return out


@dataclass
class Transfer:
    seconds: float        # first encode start .. last decode end (device time)
    raw_bytes: int        # 2 n
    sent_bytes: int       # bytes that crossed the link
    pieces: int

    @property
    def raw_gbs(self) -> float:
        return self.raw_bytes / self.seconds / 1e9

    @property
    def ratio(self) -> float:
        return self.raw_bytes / self.sent_bytes


class _Streams:
    def __init__(self, device):
        self.enc, self.send, self.recv, self.dec = (torch.cuda.Stream(device) for _ in range(4))


def send_compressed(x: torch.Tensor, codebook: torch.Tensor, chunk: int = 1024, pieces: int = 16,
                    link: str = "host", out: torch.Tensor | None = None) -> tuple[torch.Tensor, Transfer]:
    """Encode ``x`` piece by piece, move each compressed piece over ``link``
    and decode it into ``out`` (a new tensor when None). Returns the decoded
    tensor (bit-identical to ``x``) and the device-timed transfer."""
    if link not in ("host", "d2d"):
        raise ValueError("link must be 'host' or 'd2d'")
    v = _flat16(x).reshape(-1)
    dev = v.device
    n = v.numel()
    y = torch.empty_like(v) if out is None else _flat16(out).reshape(-1)
    parts = split_points(n, pieces)
    L = load()
    st = _Streams(dev)
    caps = [max_compressed_size(e - s, chunk) for s, e in parts]
    enc_buf = [torch.empty(c, dtype=torch.uint8, device=dev) for c in caps]
    rcv_buf = [torch.empty(c, dtype=torch.uint8, device=dev) for c in caps]
    host_buf = [torch.empty(c, dtype=torch.uint8, pin_memory=True) for c in caps] if link == "host" else None
    sizes = torch.zeros(max(len(parts), 1), dtype=torch.int64, device=dev)  # bytes each piece sent
    wsz = max([workspace_bytes(e - s, chunk) for s, e in parts] + [16])
    ws = torch.empty(wsz, dtype=torch.uint8, device=dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    hdr = torch.empty((max(len(parts), 1), 64), dtype=torch.uint8, pin_memory=True) if link == "host" else None
    totals = [0] * len(parts)

    def ship_host(k: int) -> None:
        # Copy engines need the length on the host: read piece k's header
        # (copied behind its encode) while piece k + 1 is already encoding.
        encoded[k].synchronize()
        nb = int.from_bytes(bytes(hdr[k, 48:56].numpy()), "little")
        totals[k] = nb
        st.send.wait_event(encoded[k])
        with torch.cuda.stream(st.send):
            host_buf[k][:nb].copy_(enc_buf[k][:nb], non_blocking=True)
            sent = torch.cuda.Event()
            sent.record(st.send)
        st.recv.wait_event(sent)
        with torch.cuda.stream(st.recv):
            rcv_buf[k][:nb].copy_(host_buf[k][:nb], non_blocking=True)
            received = torch.cuda.Event()
            received.record(st.recv)
        st.dec.wait_event(received)
        s, e = parts[k]
        check(L.uzip_decode(_p(rcv_buf[k]), nb, _p(y[s:e]), e - s, None, ctypes.c_void_p(st.dec.cuda_stream)),
              "uzip_decode")

    encoded = [torch.cuda.Event() for _ in parts]
    torch.cuda.current_stream(dev).synchronize()
    start.record(st.enc)
    for s_ in (st.send, st.recv, st.dec):
        s_.wait_event(start)
    for k, (s, e) in enumerate(parts):
        # The encodes share one workspace: they run in order on one stream.
        check(L.uzip_encode(_p(v[s:e]), e - s, chunk, _p(codebook), _p(enc_buf[k]), caps[k], _p(ws), ws.numel(),
                            None, ctypes.c_void_p(st.enc.cuda_stream)), "uzip_encode")
        if link == "host":
            with torch.cuda.stream(st.enc):
                hdr[k].copy_(enc_buf[k][:64], non_blocking=True)
            encoded[k].record(st.enc)
            if k >= 1:
                ship_host(k - 1)
            continue
        # d2d: the copy kernel reads the length on the device; nothing waits on the host.
        encoded[k].record(st.enc)
        st.send.wait_event(encoded[k])
        stream_copy(enc_buf[k], rcv_buf[k], caps[k], copied=sizes[k:k + 1], stream=st.send)
        received = torch.cuda.Event()
        received.record(st.send)
        st.dec.wait_event(received)
        check(L.uzip_decode(_p(rcv_buf[k]), caps[k], _p(y[s:e]), e - s, None,
                            ctypes.c_void_p(st.dec.cuda_stream)), "uzip_decode")
    if link == "host" and parts:
        ship_host(len(parts) - 1)
    for s_ in (st.enc, st.send, st.recv):
        st.dec.wait_stream(s_)
    stop.record(st.dec)
    stop.synchronize()
    if link == "host":
        sizes[:len(parts)] = torch.tensor(totals, dtype=torch.int64)
    sent_bytes = int(sizes[:len(parts)].sum().item())
    return y.view(x.shape) if out is None else out, Transfer(start.elapsed_time(stop) * 1e-3, 2 * n,
                                                             sent_bytes, len(parts))


def send_raw(x: torch.Tensor, pieces: int = 16, link: str = "host", out: torch.Tensor | None = None):
    """The same pipeline without the codec: each raw piece crosses the link."""
    v = _flat16(x).reshape(-1)
    dev = v.device
    n = v.numel()
    y = torch.empty_like(v) if out is None else _flat16(out).reshape(-1)
    parts = split_points(n, pieces)
    st = _Streams(dev)
    host = torch.empty(n, dtype=v.dtype, pin_memory=True) if link == "host" else None
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.current_stream(dev).synchronize()
    start.record(st.send)
    st.recv.wait_event(start)
    for s, e in parts:
        with torch.cuda.stream(st.send):
            if link == "host":
                host[s:e].copy_(v[s:e], non_blocking=True)
            else:
                y[s:e].copy_(v[s:e], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(st.send)
        if link == "host":
            st.recv.wait_event(ev)
            with torch.cuda.stream(st.recv):
                y[s:e].copy_(host[s:e], non_blocking=True)
    st.recv.wait_stream(st.send)
    stop.record(st.recv)
    stop.synchronize()
    return y.view(x.shape) if out is None else out, Transfer(start.elapsed_time(stop) * 1e-3, 2 * n, 2 * n,
                                                             len(parts))


def b_hide(g_enc: float, g_dec: float, ratio: float) -> float:
    """Largest link bandwidth whose transfer still hides the codec (appendix B)."""
    return min(g_enc, g_dec) / ratio


def model_seconds(raw_bytes: int, g_enc: float, g_dec: float, ratio: float, link_bw: float, pieces: int) -> float:
    """Appendix B's steady state (the slowest stage) plus the pipeline's fill
    and drain (one piece through the two other stages)."""
    t_enc, t_dec = raw_bytes / g_enc, raw_bytes / g_dec
    t_xfer = raw_bytes / (ratio * link_bw)
    stages = [t_enc, t_xfer, t_dec]
    slow = max(stages)
    return slow + (sum(stages) - slow) / max(pieces, 1)
