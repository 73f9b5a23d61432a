#!/usr/bin/env python3
"""Benchmark of the SplitZip BF16 codec on GB300.

One step = the whole hot path once over the KV-cache-shaped workload
(64 layers x {K,V} x 8 KV heads x 2048 tokens x 128 head dim = 268,435,456
BF16 values, chunk 1024): calibrate the Top-16 codebook on a 1 Mi-value
sample, encode the tensor, decode the stream. ``value`` is raw BF16 bytes per
second through that step; encode-only and decode-only rates, the compression
ratio and the roofline of the dominant kernel are reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the plain CPU oracle (the only other
implementation of this codec) on the host cores over a bounded slice of the
same workload. Under torchrun (N > 1) every rank runs an independent replica
on its own GPU (weak scaling, no collective on the data path); rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "encode/decode GB/s (raw BF16 bytes) @256M elems; ratio; % of HBM peak"
WORKLOAD = "kv_cache [64,2,8,2048,128] bf16 = 268,435,456 values, chunk 1024, calibration sample 1 Mi values"
CHUNK = 1024
FALLBACK_HBM_GBS = 6800.0
# Kernels one step launches: calibrate (a one-block clear of the histogram
# totals, then the histogram kernel whose last block selects the Top-16),
# encode (a one-block clear of the segment totals, dense pass, escape pass),
# decode (one kernel).
KERNELS_PER_STEP = 6


# ------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    import torch.distributed as dist

    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(v: float, device=None) -> float:
    """Largest value of v over all ranks (v itself on a single process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, device=None) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler for the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i + 1].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(path))
        return float(j["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


def source_code_hash(*paths: str) -> str:
    """First 16 hex digits of the SHA-256 of CUDA sources (in order) with
    their comments and whitespace removed: the code a profile was taken on,
    unaffected by edits to comments."""
    h = hashlib.sha256()
    for path in paths:
        text = open(path, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


def kernel_code_hash(source: str) -> str:
    """Code hash of one kernel source of the library together with the two
    headers every kernel source includes."""
    return source_code_hash(os.path.join(ROOT, "lossless_bf16_exponent_gb300", "csrc", source),
                            os.path.join(ROOT, "lossless_bf16_exponent_gb300", "csrc", "uzip_internal.cuh"),
                            os.path.join(ROOT, "include", "uzip.h"))


def profile_traffic(kernel: str, key: str = "dram_bytes_per_full_launch"):
    """DRAM bytes per launch (or, with key="dram_read_bytes_per_full_launch",
    the read bytes alone) from the committed ncu summary, if it was taken on
    the current kernel code (else None)."""
    src = {"encode": "encode.cu", "decode": "decode.cu"}[kernel]
    path = os.path.join(ROOT, "profiles", f"{kernel}_kv_cache.md")
    try:
        text = open(path).read()
        sha = kernel_code_hash(src)
        m_sha = re.search(r"code_sha256_16:\s*([0-9a-f]+)", text)
        m_b = re.search(key + r":\s*([0-9]+)", text)
        if m_sha and m_b and m_sha.group(1) == sha:
            return int(m_b.group(1))
    except OSError:
        pass
    return None


def host_threads() -> int:
    """Host cores this process may run on (the chunk-parallel oracle uses one
    thread per core)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def chunk_slices(n: int, parts: int, chunk: int = CHUNK):
    """Cut [0, n) into at most `parts` slices at chunk boundaries."""
    per = -(-n // parts)
    per = -(-per // chunk) * chunk
    return [(a, min(n, a + per)) for a in range(0, n, per)]


def oracle_parallel(o, xh, exps, threads: int):
    """The unchanged oracle on all host cores: the values cut at chunk
    boundaries into one slice per thread, each slice encoded and decoded as a
    stream of its own (as the pipeline's pieces are); ctypes releases the GIL
    for the C calls. Returns the decoded slices (for the check afterwards)."""
    from concurrent.futures import ThreadPoolExecutor

    def work(ab):
        a, b = ab
        rc, s = o.encode(xh[a:b], exps, CHUNK)
        rc2, y = o.decode(s, b - a)
        assert rc == 0 and rc2 == 0
        return y

    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(work, chunk_slices(xh.size, threads)))


def kv_input(args, dev):
    """The KV-cache workload (tensor, calibration sample): the benchmark's
    268,435,456 values at --tokens 2048, else a smaller cache of the same law
    (profiling cases)."""
    import lossless_bf16_exponent_gb300.workloads as W

    if args.tokens == W.KV_SHAPE[3]:
        return W.workload(2, device=dev)
    shape = W.KV_SHAPE[:3] + (args.tokens,) + W.KV_SHAPE[4:]
    return W.kv_cache(shape, device=dev).reshape(-1), W.kv_cache_sample(device=dev)


def kv_label(args, n: int) -> str:
    return WORKLOAD if n == 268435456 else f"kv_cache tokens={args.tokens} ({n} values), chunk {CHUNK}"


# ------------------------------------------------------------ our (GPU) arm

def run_ours(args):
    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W
    from lossless_bf16_exponent_gb300 import build as B

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    if rank == 0 and B.stale():
        B.build()
    barrier()
    uz.load()

    x, sample = kv_input(args, dev)
    n = x.numel()
    raw = 2 * n
    cb = uz.new_codebook(dev)
    out = torch.empty(uz.max_compressed_size(n, CHUNK), dtype=torch.uint8, device=dev)
    wsb = torch.empty(uz.workspace_bytes(n, CHUNK), dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev: ev[0].record(stream)
        uz.calibrate(sample, codebook=cb)
        if ev: ev[1].record(stream)
        uz.encode(x, cb, CHUNK, out=out, workspace=wsb, sync=False)
        if ev: ev[2].record(stream)
        uz.decode(out, n, out=y)
        if ev: ev[3].record(stream)

    # correctness first (bit-exact round trip), then warm-up
    step()
    info = uz.stream_info(out)
    assert info["status"] == 0, info
    assert torch.equal(y.view(torch.int16), x.view(torch.int16)), "round trip is not bit-exact"
    nbytes, m = int(info["total_bytes"]), int(info["escapes"])
    for _ in range(args.warmup):
        step()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = t0.elapsed_time(t1)
    # The timed steps may be over before nvidia-smi samples once: the same
    # step runs on for --clock-loop seconds more, still sampled, so the clock
    # record covers these kernels under load (steps and ms_per_step are not
    # touched).
    loop_steps = int(args.clock_loop * 1e3 / max(elapsed_ms / args.steps, 1e-3))
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(loop_steps):
        step()
    l1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if rank == 0 else {}
    if rank == 0 and clocks.get("samples") and loop_steps:
        loop_ms = l0.elapsed_time(l1) / loop_steps
        clocks["loaded_loop"] = {"steps": loop_steps, "seconds": round(loop_steps * loop_ms / 1e3, 2),
                                 "ms_per_step": round(loop_ms, 4),
                                 "ms_x_sm_mhz": round(loop_ms * clocks["sm_mhz"], 1)}
    cal_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    enc_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    dec_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    median_us = {op: round(statistics.median(e[i].elapsed_time(e[i + 1]) for e in evs) * 1e3, 2)
                 for i, op in enumerate(("calibrate", "encode", "decode"))}
    max_ms = max_over_ranks(elapsed_ms, dev)
    total_raw = sum_over_ranks(raw * args.steps, dev)

    if args.no_e2e:
        e2e = None
    else:
        e2e = e2e_measure(args, x, sample, cb, out, wsb, y, n, raw, stream, dev)

    cpu = cpu_baseline(x, sample) if (rank == 0 and ws == 1 and not args.no_cpu_baseline) else None
    return report(args, ws, rank, n, raw, nbytes, m, max_ms, total_raw, cal_ms, enc_ms, dec_ms, e2e, cpu,
                  clocks, sample, median_us)


def e2e_measure(args, x, sample, cb, out, wsb, y, n, raw, stream, dev):
    """Same step through the public API from pinned host buffers: every step
    copies the tensor and the sample host -> device, calibrates, encodes,
    decodes and copies the decoded tensor device -> host. Steps are pipelined
    on three streams (copy in, compute, copy out) with two device copies of
    the input and output tensors, so step k's copy out overlaps step k+1's copy
    in; the host link, not the codec, sets the pace."""
    import torch

    import lossless_bf16_exponent_gb300 as uz

    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xh.copy_(x)
    sh = torch.empty(sample.shape, dtype=sample.dtype, pin_memory=True)
    sh.copy_(sample)
    yh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xd = [torch.empty_like(x) for _ in range(2)]
    sd = [torch.empty_like(sample) for _ in range(2)]
    yd = [y, torch.empty_like(y)]
    s_in, s_c, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    computed = [None, None]   # event: compute of the last step using slot b is done
    copied_out = [None, None]  # event: copy out of the last step using slot b is done

    def e2e_step(k):
        b = k % 2
        if computed[b] is not None:
            s_in.wait_event(computed[b])  # slot b's input no longer read
        with torch.cuda.stream(s_in):
            xd[b].copy_(xh, non_blocking=True)
            sd[b].copy_(sh, non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(s_in)
        s_c.wait_event(arrived)
        if copied_out[b] is not None:
            s_c.wait_event(copied_out[b])  # slot b's output already read back
        with torch.cuda.stream(s_c):
            uz.calibrate(sd[b], codebook=cb)
            uz.encode(xd[b], cb, CHUNK, out=out, workspace=wsb, sync=False)
            uz.decode(out, n, out=yd[b])
            computed[b] = torch.cuda.Event()
            computed[b].record(s_c)
        s_out.wait_event(computed[b])
        with torch.cuda.stream(s_out):
            yh.copy_(yd[b], non_blocking=True)
            copied_out[b] = torch.cuda.Event()
            copied_out[b].record(s_out)

    e2e_steps = max(3, min(args.steps, 50))
    for k in range(max(3, args.warmup)):
        e2e_step(k)
    barrier()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for st in (s_in, s_c, s_out):
        st.wait_event(a)
    for k in range(e2e_steps):
        e2e_step(k)
    for st in (s_in, s_c, s_out):
        done = torch.cuda.Event()
        done.record(st)
        stream.wait_event(done)
    e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(e), dev)
    assert torch.equal(yh.view(torch.int16), xh.view(torch.int16)), "e2e round trip is not bit-exact"
    e2e_raw = sum_over_ranks(raw * e2e_steps, dev)
    return {"value": round(e2e_raw / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": raw + 2 * sample.numel(), "d2h_bytes_per_step": raw, "steps": e2e_steps,
            "pipeline": "copy in / compute / copy out on three streams, two device buffers"}


def report(args, ws, rank, n, raw, nbytes, m, max_ms, total_raw, cal_ms, enc_ms, dec_ms, e2e, cpu, clocks,
           sample, median_us=None):
    """The JSON line. Per-op times (calibrate_us, encode_us, decode_us and
    the rates and fractions derived from them) are means over the timed
    steps, as the page reports them; ``median_us`` holds the medians."""
    if rank != 0:
        return None
    peak, peak_src = measured_peak()
    enc_bytes = raw + nbytes  # read the BF16 tensor, write the stream
    dec_bytes = nbytes + raw  # read the stream, write the BF16 tensor
    enc_gbs = enc_bytes / (enc_ms * 1e-3) / 1e9
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    dominant = "encode" if enc_ms >= dec_ms else "decode"
    dom_gbs = enc_gbs if dominant == "encode" else dec_gbs
    line = {
        "metric": METRIC,
        "value": round(total_raw / (max_ms * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u16",
        "data": "synthetic",
        "config": {"workload": kv_label(args, n),
                   "step": "calibrate + encode + decode",
                   "l2": "inputs larger than L2 (512 MiB BF16 tensor, 403 MB stream)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "encode_gbs_raw": round(raw / (enc_ms * 1e-3) / 1e9, 1),
        "decode_gbs_raw": round(raw / (dec_ms * 1e-3) / 1e9, 1),
        "calibrate_us": round(cal_ms * 1e3, 2),
        "encode_us": round(enc_ms * 1e3, 2),
        "decode_us": round(dec_ms * 1e3, 2),
        "median_us": median_us,
        "ratio": round(raw / nbytes, 5),
        "ratio_payload": round(raw / (n + (n + 1) // 2 + 3 * m), 5),
        "escape_rate": m / n,
        "hbm": {"encode": {"gbs": round(enc_gbs, 1), "frac": round(enc_gbs / peak, 4)},
                "decode": {"gbs": round(dec_gbs, 1), "frac": round(dec_gbs / peak, 4)},
                "peak_gbs": peak, "peak_source": peak_src, "vs_8tbs": {
                    "encode": round(enc_gbs / 8000, 4), "decode": round(dec_gbs / 8000, 4)}},
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": round(dom_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(dom_gbs / peak, 4), "peak_source": peak_src,
                     "traffic": profile_traffic(dominant),
                     "algorithmic_bytes": enc_bytes if dominant == "encode" else dec_bytes,
                     # DRAM writes still in L2 when a kernel ends are not counted in its
                     # traffic, so the reads are the check for wasted traffic
                     "traffic_read": profile_traffic(dominant, "dram_read_bytes_per_full_launch"),
                     "algorithmic_read_bytes": raw if dominant == "encode" else nbytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clocks,
    }
    return line


def cpu_baseline(x, sample, budget_s: float = 8.0):
    """The oracle, as it stands, on the host: calibrate on the sample, encode
    and decode the whole workload, repeated while the budget lasts -- on all
    host cores (one chunk-aligned slice per thread, the unchanged oracle in
    each) and, beside it, on one thread."""
    import numpy as np

    import lossless_bf16_exponent_gb300.workloads as W
    import oracle

    o = oracle.Oracle()
    xh, sh = W.as_u16(x), W.as_u16(sample)
    threads = host_threads()

    def timed(parallel: bool):
        t_total, raw_total, reps = 0.0, 0, 0
        while reps < 1 or (t_total < budget_s and reps < 5):
            t = time.perf_counter()
            exps = o.calibrate(sh)
            if parallel:
                ys = oracle_parallel(o, xh, exps, threads)
            else:
                rc, s = o.encode(xh, exps, CHUNK)
                rc2, y = o.decode(s, xh.size)
                assert rc == 0 and rc2 == 0
                ys = [y]
            t_total += time.perf_counter() - t
            assert np.array_equal(np.concatenate(ys), xh)
            raw_total += 2 * xh.size
            reps += 1
        return raw_total / t_total / 1e9, reps, t_total

    par, reps_p, t_p = timed(True)
    one, reps_1, t_1 = timed(False)
    return {"value": round(par, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"whole workload ({xh.size} values) x{reps_p}: calibrate 1 Mi sample, then encode + "
                      f"decode of {threads} chunk-aligned slices on {threads} threads, {t_p:.1f} s",
            "single_thread": {"value": round(one, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"whole workload x{reps_1} on one thread, {t_1:.1f} s"}}


# ------------------------------------------------------ reference (oracle) arm

def run_reference(args):
    """The oracle alone on the host cores (all of them, one chunk-aligned
    slice per thread), each step calibrating on the sample and encoding and
    decoding a slice of the workload sized so the whole run stays within
    about two minutes -- the whole workload when that fits."""
    import numpy as np
    import torch

    import lossless_bf16_exponent_gb300.workloads as W
    import oracle

    ws, rank, local = dist_env()
    if rank != 0:
        return None  # rank 0 alone runs the CPU reference
    o = oracle.Oracle()
    threads = host_threads()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x, sample = W.workload(2, device=dev)
    xh, sh = W.as_u16(x), W.as_u16(sample)
    del x
    probe = xh[: 1 << 24]
    t = time.perf_counter()
    oracle_parallel(o, probe, o.calibrate(sh), threads)
    per_val = (time.perf_counter() - t) / probe.size
    steps_total = args.steps + args.warmup
    n_slice = int(min(xh.size, max(1 << 20, 110.0 / max(steps_total, 1) / per_val)))
    if n_slice < xh.size:  # a slice of whole chunks, at chunk-aligned offsets
        n_slice = max(8192, n_slice - n_slice % 8192)
    times = []
    for k in range(steps_total):
        off = (k * n_slice) % (xh.size - n_slice + 1) // 8192 * 8192
        sl = xh[off:off + n_slice]
        t = time.perf_counter()
        exps = o.calibrate(sh)
        ys = oracle_parallel(o, sl, exps, threads)
        dt = time.perf_counter() - t
        assert np.array_equal(np.concatenate(ys), sl)
        if k >= args.warmup:
            times.append(dt)
    elapsed = sum(times)
    value = 2 * n_slice * len(times) / elapsed / 1e9
    whole = n_slice == xh.size
    what = "the whole workload" if whole else f"a slice of {n_slice} of its {xh.size} values"
    sample_txt = (f"{what} per step (calibrate 1 Mi sample, then encode + decode of {threads} chunk-aligned "
                  f"slices on {threads} threads)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed / len(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "step": "calibrate + encode + decode (CPU oracle, " + ("whole workload" if whole else
                                                                       "bounded slice") + ")"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample_txt},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------ next rows

def run_dynamic(args):
    """Per-input codebook (SplitZip review page, §4.3 Table 7): every step
    builds the codebook from the whole tensor and encodes with it
    (uzip_encode_dynamic); the page's dynamic variant ran at 80.7 GB/s
    encode on an H200 against 613.3 GB/s with the offline codebook."""
    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    x, sample = kv_input(args, dev)
    n = x.numel()
    raw = 2 * n
    cb = uz.new_codebook(dev)
    out = torch.empty(uz.max_compressed_size(n, CHUNK), dtype=torch.uint8, device=dev)
    wsb = torch.empty(uz.workspace_bytes(n, CHUNK), dtype=torch.uint8, device=dev)
    stream, nbytes, _ = uz.encode_dynamic(x, CHUNK, codebook=cb, out=out, workspace=wsb)
    y = uz.decode(out, n, stream_bytes=nbytes)
    assert torch.equal(y.view(torch.int16), x.view(torch.int16)), "round trip is not bit-exact"
    del y
    for _ in range(args.warmup):
        uz.encode_dynamic(x, CHUNK, codebook=cb, out=out, workspace=wsb, sync=False)
    st = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier()
    torch.cuda.synchronize()
    ev[0].record(st)
    for _ in range(args.steps):
        uz.encode_dynamic(x, CHUNK, codebook=cb, out=out, workspace=wsb, sync=False)
    ev[1].record(st)
    torch.cuda.synchronize()
    ms = max_over_ranks(ev[0].elapsed_time(ev[1]), dev) / args.steps
    # offline-codebook encode of the same tensor, for the ratio the page quotes
    ucb = uz.calibrate(sample)
    for _ in range(args.warmup):
        uz.encode(x, ucb, CHUNK, out=out, workspace=wsb, sync=False)
    torch.cuda.synchronize()
    ev[0].record(st)
    for _ in range(args.steps):
        uz.encode(x, ucb, CHUNK, out=out, workspace=wsb, sync=False)
    ev[1].record(st)
    torch.cuda.synchronize()
    ms_static = ev[0].elapsed_time(ev[1]) / args.steps
    if rank != 0:
        return None
    peak, peak_src = measured_peak()
    alg = 2 * raw + nbytes  # histogram pass reads the tensor, encode reads it again and writes the stream
    return {
        "mode": "dynamic", "metric": "dynamic Top-16 encode GB/s (raw BF16 bytes) @256M elems",
        "value": round(raw * ws / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u16", "data": "synthetic",
        "config": {"workload": kv_label(args, n), "codebook": "Top-16 of the whole tensor, rebuilt every step"},
        "roofline": {"kernel": "calibrate + encode", "bound": "hbm", "achieved": round(alg / (ms * 1e-3) / 1e9, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(alg / (ms * 1e-3) / 1e9 / peak, 4),
                     "peak_source": peak_src, "algorithmic_bytes": alg},
        "static_encode_us": round(ms_static * 1e3, 2), "dynamic_encode_us": round(ms * 1e3, 2),
        "slowdown_vs_static": round(ms / ms_static, 3), "ratio": round(raw / nbytes, 5),
        "page_h200": {"dynamic_encode_gbs": 80.7, "static_encode_gbs": 613.3, "slowdown": 7.6},
    }


def run_pipeline(args):
    """Streamed transfer (SplitZip review page, appendix B): the 256M KV tensor
    in pieces through encode -> link -> decode, against the same pipeline
    moving raw pieces, on two links (pinned host memory over NVLink-C2C; a
    device-to-device copy), with B_hide = min(G_enc, G_dec) / rho and the
    appendix's stage model next to the measured times."""
    import statistics as stats

    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W
    from lossless_bf16_exponent_gb300 import pipeline as PL

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    x, sample = kv_input(args, dev)
    n = x.numel()
    raw = 2 * n
    cb = uz.calibrate(sample)
    out = torch.empty(uz.max_compressed_size(n, CHUNK), dtype=torch.uint8, device=dev)
    wsb = torch.empty(uz.workspace_bytes(n, CHUNK), dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    _, nbytes = uz.encode(x, cb, CHUNK, out=out, workspace=wsb)
    ratio = raw / nbytes
    st = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    te, td = [], []
    for k in range(args.warmup + 20):
        ev[0].record(st)
        uz.encode(x, cb, CHUNK, out=out, workspace=wsb, sync=False)
        ev[1].record(st)
        uz.decode(out, n, out=y, stream_bytes=nbytes)
        ev[2].record(st)
        torch.cuda.synchronize()
        if k >= args.warmup:
            te.append(ev[0].elapsed_time(ev[1]))
            td.append(ev[1].elapsed_time(ev[2]))
    g_enc = raw / (stats.median(te) * 1e-3)
    g_dec = raw / (stats.median(td) * 1e-3)
    pieces = 16
    runs = max(3, min(args.steps, 10))
    links = {}
    for link in ("host", "d2d"):
        res = {}
        for name, fn in (("raw", lambda: PL.send_raw(x, pieces=pieces, link=link, out=y)),
                         ("compressed", lambda: PL.send_compressed(x, cb, CHUNK, pieces=pieces, link=link, out=y))):
            fn()  # warm-up (allocations, first touch of pinned memory)
            secs = []
            for _ in range(runs):
                yy, tr = fn()
                secs.append(tr.seconds)
            assert torch.equal(y.view(torch.int16), x.view(torch.int16)), f"{link} {name}: not bit-exact"
            res[name] = {"seconds": stats.median(secs), "raw_gbs": round(raw / stats.median(secs) / 1e9, 2),
                         "sent_bytes": tr.sent_bytes}
        b_link = raw / res["raw"]["seconds"]  # the link's own rate, from the raw pipeline
        model = PL.model_seconds(raw, g_enc, g_dec, ratio, b_link, pieces)
        links[link] = {
            "raw_pipeline_gbs": res["raw"]["raw_gbs"], "compressed_pipeline_gbs": res["compressed"]["raw_gbs"],
            "speedup": round(res["raw"]["seconds"] / res["compressed"]["seconds"], 3),
            "link_gbs": round(b_link / 1e9, 1), "codec_hidden": bool(b_link <= PL.b_hide(g_enc, g_dec, ratio)),
            "model_us": round(model * 1e6, 1), "measured_us": round(res["compressed"]["seconds"] * 1e6, 1),
            "sent_bytes": res["compressed"]["sent_bytes"],
        }
    if rank != 0:
        return None
    return {
        "mode": "pipeline", "metric": "compressed transfer GB/s (raw BF16 bytes through encode -> link -> decode)",
        "value": links["host"]["compressed_pipeline_gbs"], "unit": "GB/s", "n_gpus": ws, "steps": runs,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
        "data": "synthetic", "config": {"workload": kv_label(args, n), "pieces": pieces, "value_link": "host"},
        "g_enc_gbs": round(g_enc / 1e9, 1), "g_dec_gbs": round(g_dec / 1e9, 1), "ratio": round(ratio, 5),
        "b_hide_gbs": round(PL.b_hide(g_enc, g_dec, ratio) / 1e9, 1), "links": links,
        "note": ("the stage model assumes independent resources; the host link is one (copy engines over "
                 "NVLink-C2C), the d2d link is not (its copies share HBM and SMs with the codec kernels)"),
        "page_h200": {"b_hide_gbs": 463.2, "g_enc_gbs": 613.3, "g_dec_gbs": 2181.8, "ratio": 1.324},
    }


def run_chunks(args):
    """Escape-capture chunk size (SplitZip review page, appendix D, Fig. 6):
    the same KV tensor encoded with chunks of 256 .. 65536 values. The chunk
    sets how many 16-bit escape positions share one 4-byte offset: small
    chunks cost offset bytes, large chunks cost nothing in bytes but make
    each decode tile walk longer escape blocks."""
    import statistics as stats

    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    x, sample = kv_input(args, dev)
    n = x.numel()
    raw = 2 * n
    cb = uz.calibrate(sample)
    y = torch.empty_like(x)
    st = torch.cuda.current_stream(dev)
    rows = []
    for chunk in (256, 512, 1024, 2048, 4096, 16384, 65536):
        out = torch.empty(uz.max_compressed_size(n, chunk), dtype=torch.uint8, device=dev)
        wsb = torch.empty(uz.workspace_bytes(n, chunk), dtype=torch.uint8, device=dev)
        _, nbytes = uz.encode(x, cb, chunk, out=out, workspace=wsb)
        info = uz.stream_info(out, nbytes)
        reps = max(5, min(args.steps, 50))
        for _ in range(args.warmup):
            uz.encode(x, cb, chunk, out=out, workspace=wsb, sync=False)
            uz.decode(out, n, out=y, stream_bytes=nbytes)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        torch.cuda.synchronize()
        for ev in evs:  # back to back, as in the benchmark step
            ev[0].record(st)
            uz.encode(x, cb, chunk, out=out, workspace=wsb, sync=False)
            ev[1].record(st)
            uz.decode(out, n, out=y, stream_bytes=nbytes)
            ev[2].record(st)
        torch.cuda.synchronize()
        te = [ev[0].elapsed_time(ev[1]) for ev in evs]
        td = [ev[1].elapsed_time(ev[2]) for ev in evs]
        assert torch.equal(y.view(torch.int16), x.view(torch.int16)), f"chunk {chunk}: not bit-exact"
        m = int(info["escapes"])
        nc = -(-n // chunk)
        rows.append({"chunk": chunk, "stream_bytes": nbytes, "ratio": round(raw / nbytes, 5),
                     "payload_ratio": round(raw / (n + (n + 1) // 2 + 3 * m), 5), "offset_bytes": 4 * (nc + 1),
                     "encode_us": round(stats.median(te) * 1e3, 2), "decode_us": round(stats.median(td) * 1e3, 2),
                     "encode_gbs_raw": round(raw / (stats.median(te) * 1e-3) / 1e9, 1),
                     "decode_gbs_raw": round(raw / (stats.median(td) * 1e-3) / 1e9, 1)})
        del out, wsb
    if rank != 0:
        return None
    best = next(r for r in rows if r["chunk"] == CHUNK)
    return {"mode": "chunks", "metric": "encode/decode GB/s and ratio vs escape chunk size @256M elems",
            "value": best["decode_gbs_raw"], "unit": "GB/s", "n_gpus": ws, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": kv_label(args, n), "value": "decode GB/s at chunk 1024"}, "rows": rows}


def run_e5m2(args):
    """FP8 E5M2 codec (SplitZip review page, §4.2 / appendix C: the Top-16
    framework on E5M2 KV, a further 1.14x): the KV-cache law quantised to
    E5M2 (268,435,456 one-byte values), encode and decode timed back to back."""
    import statistics as stats

    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    xb, sb = kv_input(args, dev)  # the KV law, quantised to E5M2 as an FP8 KV cache stores it
    x, sample = W.to_e5m2_bits(xb), W.to_e5m2_bits(sb)
    del xb
    n = x.numel()
    cb = uz.e5m2_calibrate(sample)
    out = torch.empty(uz.e5m2_compressed_size(n, n, CHUNK), dtype=torch.uint8, device=dev)
    wsb = torch.empty(uz.workspace_bytes(n, CHUNK), dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    _, nbytes = uz.e5m2_encode(x, cb, CHUNK, out=out, workspace=wsb)
    uz.e5m2_decode(out, n, out=y, stream_bytes=nbytes)
    assert torch.equal(y, x), "E5M2 round trip is not bit-exact"
    m = int.from_bytes(bytes(out[24:32].cpu().numpy()), "little")
    st = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        uz.e5m2_encode(x, cb, CHUNK, out=out, workspace=wsb, sync=False)
        uz.e5m2_decode(out, n, out=y, stream_bytes=nbytes)
    reps = max(10, min(args.steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    barrier()
    torch.cuda.synchronize()
    for ev in evs:
        ev[0].record(st)
        uz.e5m2_encode(x, cb, CHUNK, out=out, workspace=wsb, sync=False)
        ev[1].record(st)
        uz.e5m2_decode(out, n, out=y, stream_bytes=nbytes)
        ev[2].record(st)
    torch.cuda.synchronize()
    te = stats.mean(e[0].elapsed_time(e[1]) for e in evs)
    td = stats.mean(e[1].elapsed_time(e[2]) for e in evs)
    step_ms = max_over_ranks(evs[0][0].elapsed_time(evs[-1][2]) / reps, dev)
    if rank != 0:
        return None
    peak, peak_src = measured_peak()
    alg = n + nbytes
    enc_gbs, dec_gbs = alg / (te * 1e-3) / 1e9, alg / (td * 1e-3) / 1e9
    dom, gbs = ("encode", enc_gbs) if te >= td else ("decode", dec_gbs)
    return {
        "mode": "e5m2", "metric": "E5M2 encode/decode GB/s (raw FP8 bytes) @256M elems; ratio",
        "value": round(n * ws / (step_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": ws, "steps": reps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": kv_label(args, n) + ", quantised to FP8 E5M2",
                   "step": "encode + decode"},
        "encode_us": round(te * 1e3, 2), "decode_us": round(td * 1e3, 2),
        "encode_gbs_raw": round(n / (te * 1e-3) / 1e9, 1), "decode_gbs_raw": round(n / (td * 1e-3) / 1e9, 1),
        "ratio": round(n / nbytes, 5), "escape_rate": m / n, "page_ratio": 1.14,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_source": peak_src, "algorithmic_bytes": alg},
    }


def run_sentinel(args):
    """Top-15 + sentinel against Top-16 with explicit positions (SplitZip
    review page, §3.4 and Table 6): the same KV tensor and calibration sample,
    the sentinel codebook made from the Top-16 one's first 15 exponents, each
    codec's encode and decode timed back to back; ratio of each stream."""
    import statistics as stats

    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    x, sample = kv_input(args, dev)
    n = x.numel()
    raw = 2 * n
    cb16 = uz.calibrate(sample)
    cb15 = uz.make_sentinel(cb16.clone())
    out = torch.empty(uz.max_compressed_size(n, CHUNK), dtype=torch.uint8, device=dev)
    wsb = torch.empty(uz.workspace_bytes(n, CHUNK), dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    st = torch.cuda.current_stream(dev)
    codecs = {
        "top16": (lambda: uz.encode(x, cb16, CHUNK, out=out, workspace=wsb, sync=False),
                  lambda nb: uz.decode(out, n, out=y, stream_bytes=nb)),
        "top15_sentinel": (lambda: uz.sentinel_encode(x, cb15, CHUNK, out=out, workspace=wsb, sync=False),
                           lambda nb: uz.sentinel_decode(out, n, out=y, stream_bytes=nb)),
    }
    reps = max(10, min(args.steps, 200))
    res = {}
    for name, (enc, dec) in codecs.items():
        enc()
        info = uz.stream_info(out)
        nbytes = int(info["total_bytes"])
        dec(nbytes)
        torch.cuda.synchronize()
        assert info["status"] == 0 and torch.equal(y.view(torch.int16), x.view(torch.int16)), name
        for _ in range(args.warmup):
            enc()
            dec(nbytes)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        barrier()
        torch.cuda.synchronize()
        for ev in evs:
            ev[0].record(st)
            enc()
            ev[1].record(st)
            dec(nbytes)
            ev[2].record(st)
        torch.cuda.synchronize()
        te = stats.mean(e[0].elapsed_time(e[1]) for e in evs)
        td = stats.mean(e[1].elapsed_time(e[2]) for e in evs)
        m = int(info["escapes"])
        res[name] = {"stream_bytes": nbytes, "ratio": round(raw / nbytes, 5),
                     "payload_ratio": round(raw / int(info["payload_bytes"]), 5), "escapes": m,
                     "encode_us": round(te * 1e3, 2), "decode_us": round(td * 1e3, 2),
                     "encode_gbs_raw": round(raw / (te * 1e-3) / 1e9, 1),
                     "decode_gbs_raw": round(raw / (td * 1e-3) / 1e9, 1),
                     "decode_frac_of_peak": None, "_alg": raw + nbytes, "_td": td}
    if rank != 0:
        return None
    peak, peak_src = measured_peak()
    for r in res.values():
        r["decode_frac_of_peak"] = round(r.pop("_alg") / (r.pop("_td") * 1e-3) / 1e9 / peak, 4)
    s15 = res["top15_sentinel"]
    return {
        "mode": "sentinel", "metric": "Top-15+sentinel vs Top-16 decode GB/s (raw BF16 bytes) and ratio @256M elems",
        "value": s15["decode_gbs_raw"], "unit": "GB/s", "n_gpus": ws, "steps": reps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
        "config": {"workload": kv_label(args, n), "value": "Top-15 + sentinel decode GB/s", "peak_gbs": peak,
                   "peak_source": peak_src},
        "codecs": res,
        "decode_speed_top16_over_sentinel": round(res["top15_sentinel"]["decode_us"] / res["top16"]["decode_us"], 3),
        "page_table6": {"sentinel_ratio": 1.331, "sentinel_decode_gbs": 620.8, "top16_decode_speedup": 3.5},
    }


def _timed_calls(fn, reps, flush, st):
    """Device time of each of ``reps`` calls of fn, L2 flushed before each
    (the flush is outside the timed events). Returns the median in ms."""
    import statistics as stats

    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        flush.fill_(1)
        a.record(st)
        fn()
        b.record(st)
    torch.cuda.synchronize()
    return stats.median(a.elapsed_time(b) for a, b in evs)


def run_sweep(args):
    """Message-size sweep: N(0,1) BF16 buffers of 4 KiB .. 1 GiB (powers of
    two) with chunks of 256, 1024 and 4096 values, the transfer-sized
    messages of a KV-cache hand-off. Per call: device time of encode and of
    decode (median, L2 flushed before every call, so no message is served
    from L2 by its previous call) and the host time a call takes to enqueue.
    Every point is checked bit-exact first."""
    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    st = torch.cuda.current_stream(dev)
    cb = uz.calibrate(W.sweep_sample(dev))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # twice the L2
    rows = []
    for chunk in W.SWEEP_CHUNKS:
        for nbytes in W.SWEEP_BYTES:
            x = W.sweep(nbytes, dev)
            n = x.numel()
            out = torch.empty(uz.max_compressed_size(n, chunk), dtype=torch.uint8, device=dev)
            wsb = torch.empty(uz.workspace_bytes(n, chunk), dtype=torch.uint8, device=dev)
            y = torch.empty_like(x)
            _, sb = uz.encode(x, cb, chunk, out=out, workspace=wsb)
            uz.decode(out, n, out=y, stream_bytes=sb)
            assert torch.equal(y.view(torch.int16), x.view(torch.int16)), f"{nbytes} B, chunk {chunk}: not bit-exact"
            reps = 30 if nbytes <= (64 << 20) else 10
            for _ in range(args.warmup):
                uz.encode(x, cb, chunk, out=out, workspace=wsb, sync=False)
                uz.decode(out, n, out=y, stream_bytes=sb)
            te = _timed_calls(lambda: uz.encode(x, cb, chunk, out=out, workspace=wsb, sync=False), reps, flush, st)
            td = _timed_calls(lambda: uz.decode(out, n, out=y, stream_bytes=sb), reps, flush, st)
            host_us = None
            if nbytes <= (1 << 20):  # enqueue cost per call, back to back, no synchronisation
                torch.cuda.synchronize()
                t = time.perf_counter()
                for _ in range(200):
                    uz.encode(x, cb, chunk, out=out, workspace=wsb, sync=False)
                    uz.decode(out, n, out=y, stream_bytes=sb)
                host_us = round((time.perf_counter() - t) / 200 * 1e6, 2)
                torch.cuda.synchronize()
            rows.append({"bytes": nbytes, "chunk": chunk, "ratio": round(nbytes / sb, 5),
                         "encode_us": round(te * 1e3, 2), "decode_us": round(td * 1e3, 2),
                         "encode_gbs_raw": round(nbytes / (te * 1e-3) / 1e9, 2),
                         "decode_gbs_raw": round(nbytes / (td * 1e-3) / 1e9, 2),
                         "host_us_per_encode_decode": host_us})
            del x, out, wsb, y
        torch.cuda.empty_cache()
    if rank != 0:
        return None
    big = next(r for r in rows if r["bytes"] == W.SWEEP_BYTES[-1] and r["chunk"] == CHUNK)
    small = next(r for r in rows if r["bytes"] == W.SWEEP_BYTES[0] and r["chunk"] == CHUNK)
    return {"mode": "sweep", "metric": "per-call encode/decode latency (us) and GB/s (raw BF16) vs message size",
            "value": round(small["encode_us"] + small["decode_us"], 2), "unit": "us", "n_gpus": ws,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": "N(0,1) BF16, 4 KiB .. 1 GiB x chunk {256, 1024, 4096}",
                       "value": "encode + decode device time of a 4 KiB message at chunk 1024",
                       "l2": "flushed (256 MiB write) before every timed call"},
            "largest": {"bytes": big["bytes"], "encode_gbs_raw": big["encode_gbs_raw"],
                        "decode_gbs_raw": big["decode_gbs_raw"]},
            "rows": rows}


def run_workloads(args):
    """The other full-size workloads through the same calibrate -> encode ->
    decode path: rows of log-uniform scale (8192 x 128), the heavy-tailed
    escape stress (64 Mi values), the gradient-like buffer (1 Gi values, 10 %
    zeros, 1 % subnormals; encode then decode in one stream) and the KV cache
    for comparison. Device time per op (median; inputs of 128 MiB and more
    exceed L2, the 2 MiB one is flushed from L2 before every call)."""
    import torch

    import lossless_bf16_exponent_gb300 as uz
    import lossless_bf16_exponent_gb300.workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    uz.load()
    st = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    names = {1: "rows_lognormal_scale 8192x128", 2: "kv_cache 256M", 3: "heavy_tailed 64M (escape stress)",
             5: "gradient_like 1G"}
    peak, peak_src = measured_peak()
    res = {}
    for k in (args.only,) if args.only else (1, 2, 3, 5):
        x, sample = W.workload(k, device=dev)
        if args.n and k == 1:  # fewer rows of 128 (a short message: profiling cases)
            x = W.rows_lognormal_scale(max(1, args.n // 128), 128, device=dev).reshape(-1)
        elif args.n and k == 3:  # a smaller instance of the law (profiling cases)
            x = W.heavy_tailed(args.n, device=dev)
        elif args.n and k == 5:
            x = W.gradient_like(args.n, device=dev)
        n = x.numel()
        raw = 2 * n
        cb = uz.calibrate(sample)
        out = torch.empty(uz.max_compressed_size(n, CHUNK), dtype=torch.uint8, device=dev)
        wsb = torch.empty(uz.workspace_bytes(n, CHUNK), dtype=torch.uint8, device=dev)
        y = torch.empty_like(x)
        _, sb = uz.encode(x, cb, CHUNK, out=out, workspace=wsb)
        info = uz.stream_info(out, sb)
        uz.decode(out, n, out=y, stream_bytes=sb)
        assert torch.equal(y.view(torch.int16), x.view(torch.int16)), f"workload {k}: not bit-exact"
        for _ in range(args.warmup):
            uz.encode(x, cb, CHUNK, out=out, workspace=wsb, sync=False)
            uz.decode(out, n, out=y, stream_bytes=sb)
        reps = 20 if k != 5 else 10
        te = _timed_calls(lambda: uz.encode(x, cb, CHUNK, out=out, workspace=wsb, sync=False), reps, flush, st)
        td = _timed_calls(lambda: uz.decode(out, n, out=y, stream_bytes=sb), reps, flush, st)
        m = int(info["escapes"])
        res[names[k]] = {"n": n, "escape_rate": round(m / n, 6), "ratio": round(raw / sb, 5),
                         "encode_us": round(te * 1e3, 2), "decode_us": round(td * 1e3, 2),
                         "encode_gbs_raw": round(raw / (te * 1e-3) / 1e9, 1),
                         "decode_gbs_raw": round(raw / (td * 1e-3) / 1e9, 1),
                         "encode_frac": round((raw + sb) / (te * 1e-3) / 1e9 / peak, 4),
                         "decode_frac": round((raw + sb) / (td * 1e-3) / 1e9 / peak, 4)}
        del x, sample, out, wsb, y
        torch.cuda.empty_cache()
    if rank != 0:
        return None
    if args.only:
        r = res[names[args.only]]
        return {"mode": "workloads", "metric": "encode/decode GB/s (raw BF16 bytes) and ratio of one workload",
                "value": round(2 * r["n"] / ((r["encode_us"] + r["decode_us"]) * 1e-6) / 1e9, 1), "unit": "GB/s",
                "n_gpus": ws, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
                "data": "synthetic", "config": {"workload": f"{names[args.only]} ({r['n']} values), chunk 1024",
                                                "peak_gbs": peak, "peak_source": peak_src},
                "workloads": res}
    g = res[names[5]]
    return {"mode": "workloads", "metric": "encode/decode GB/s (raw BF16 bytes) and ratio per workload",
            "value": round(2 * g["n"] / ((g["encode_us"] + g["decode_us"]) * 1e-6) / 1e9, 1), "unit": "GB/s",
            "n_gpus": ws, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
            "data": "synthetic",
            "config": {"workload": "rows 8192x128, kv_cache 256M, heavy_tailed 64M, gradient_like 1G; chunk 1024",
                       "value": "gradient_like 1G: raw bytes / (encode + decode time), one stream",
                       "peak_gbs": peak, "peak_source": peak_src},
            "workloads": res}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["codec", "dynamic", "pipeline", "chunks", "e5m2", "sentinel", "sweep", "workloads"],
                    default="codec",
                    help="codec = the benchmark step; dynamic = per-input codebook encode; "
                         "pipeline = streamed compressed transfer; chunks / e5m2 / sentinel = the page's "
                         "variants; sweep = message sizes 4 KiB .. 1 GiB; workloads = the other full-size laws")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--tokens", type=int, default=2048,
                    help="tokens of the KV-cache workload (2048 = the benchmark; smaller for profiling)")
    ap.add_argument("--clock-loop", type=float, default=1.5,
                    help="seconds of sampled steps after the timed ones, for the clock record (0: none)")
    ap.add_argument("--only", type=int, choices=[1, 2, 3, 5], default=0,
                    help="workloads mode: run this workload alone")
    ap.add_argument("--n", type=int, default=0,
                    help="workloads mode: values of the row-scaled (1, rounded to rows of 128), "
                         "heavy-tailed (3) or gradient-like (5) law")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.mode == "dynamic":
        line = run_dynamic(args)
    elif args.mode == "pipeline":
        line = run_pipeline(args)
    elif args.mode == "chunks":
        line = run_chunks(args)
    elif args.mode == "e5m2":
        line = run_e5m2(args)
    elif args.mode == "sentinel":
        line = run_sentinel(args)
    elif args.mode == "sweep":
        line = run_sweep(args)
    elif args.mode == "workloads":
        line = run_workloads(args)
    else:
        line = run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
