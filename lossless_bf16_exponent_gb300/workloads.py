"""Seeded synthetic BF16 workloads.

This module only draws random tensors; it holds none of the codec's arithmetic,
so both the CUDA path and the CPU oracle can be fed from it. Every generator
takes a seed and a device and returns ``torch.bfloat16`` tensors (fp32 draws
rounded to nearest-even by ``Tensor.to``).

The SplitZip review page measures on real Qwen3-32B KV activations (§4.1),
which are not available here; the generators below are synthetic stand-ins with
the shapes and value laws of the five benchmark workloads:

1. ``rows_lognormal_scale``: 8192 x 128, row r ~ N(0, s_r^2), s_r log-uniform in
   [0.05, 4]; calibration sample 512 rows of the same law.
2. ``kv_cache``: [64 layers, 2 (K, V), 8 KV heads, 2048 tokens, 128 head dim],
   Gaussian entries scaled per (layer, head) by a log-uniform factor in
   [0.1, 8] shared by K and V, 0.1 % of the (layer, K/V, head, dim) channels
   multiplied by 20; calibration sample 1 Mi values of the same law.
3. ``heavy_tailed``: 0.5 * Student-t(3) plus 2 % of entries multiplied by 2^k,
   k uniform in [8, 20]; calibrated on pure N(0, 1).
4. ``gaussian``: N(0, 1) message-size sweep.
5. ``gradient_like``: N(0, 1e-3^2) with 10 % exact +0.0 and 1 % subnormals
   (exponent field 0, random sign, mantissa uniform in [1, 127]).

Seeds: data of workload k uses ``1000 + k`` and its calibration sample
``2000 + k`` unless the caller passes others.
"""
from __future__ import annotations

import math

import torch

DATA_SEED = 1000
CALIB_SEED = 2000

KV_SHAPE = (64, 2, 8, 2048, 128)
SWEEP_BYTES = [1 << p for p in range(12, 31)]  # 4 KiB .. 1 GiB
SWEEP_CHUNKS = (256, 1024, 4096)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(n: int, seed: int = DATA_SEED + 4, device="cpu", std: float = 1.0) -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(n, generator=g, device=device) * std).to(torch.bfloat16)


def rows_lognormal_scale(rows: int = 8192, cols: int = 128, seed: int = DATA_SEED + 1,
                         device="cpu", lo: float = 0.05, hi: float = 4.0) -> torch.Tensor:
    g = _gen(seed, device)
    u = torch.rand(rows, 1, generator=g, device=device)
    s = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    x = torch.randn(rows, cols, generator=g, device=device) * s
    return x.to(torch.bfloat16)


def kv_cache(shape=KV_SHAPE, seed: int = DATA_SEED + 2, device="cpu", lo: float = 0.1,
             hi: float = 8.0, outlier_frac: float = 0.001, outlier_gain: float = 20.0) -> torch.Tensor:
    L, KV, H, T, D = shape
    g = _gen(seed, device)
    u = torch.rand(L, 1, H, 1, 1, generator=g, device=device)
    scale = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    n_channels = L * KV * H * D
    n_out = int(round(outlier_frac * n_channels))
    pick = torch.randperm(n_channels, generator=g, device=device)[:n_out]
    gain = torch.ones(n_channels, device=device)
    gain[pick] = outlier_gain
    gain = gain.view(L, KV, H, D).unsqueeze(3)  # [L, KV, H, 1, D]
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for l in range(L):  # one layer at a time keeps the fp32 temporary small
        z = torch.randn(KV, H, T, D, generator=g, device=device)
        out[l] = (z * scale[l] * gain[l]).to(torch.bfloat16)
    return out


def kv_cache_sample(n: int = 1 << 20, seed: int = CALIB_SEED + 2, device="cpu") -> torch.Tensor:
    """Calibration sample drawn from the same law as ``kv_cache``: tokens of a
    smaller cache with the full layer/head/dim structure."""
    L, KV, H, _, D = KV_SHAPE
    t = max(1, n // (L * KV * H * D))
    x = kv_cache((L, KV, H, t, D), seed=seed, device=device).reshape(-1)
    return x[:n]


def heavy_tailed(n: int = 1 << 26, seed: int = DATA_SEED + 3, device="cpu", nu: int = 3,
                 scale: float = 0.5, frac: float = 0.02, kmin: int = 8, kmax: int = 20) -> torch.Tensor:
    g = _gen(seed, device)
    z = torch.randn(n, generator=g, device=device)
    chi2 = torch.zeros(n, device=device)
    for _ in range(nu):
        w = torch.randn(n, generator=g, device=device)
        chi2 += w * w
    t = z / torch.sqrt(chi2 / nu)
    hit = torch.rand(n, generator=g, device=device) < frac
    k = torch.randint(kmin, kmax + 1, (n,), generator=g, device=device).to(torch.float32)
    x = scale * t * torch.where(hit, torch.exp2(k), torch.ones_like(k))
    return x.to(torch.bfloat16)


def gradient_like(n: int = 1 << 30, seed: int = DATA_SEED + 5, device="cpu", std: float = 1e-3,
                  zero_frac: float = 0.10, subnormal_frac: float = 0.01) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    g = _gen(seed, device)
    step = 1 << 26
    for s in range(0, n, step):  # slices bound the temporaries at ~1.5 GiB
        m = min(step, n - s)
        gauss = (torch.randn(m, generator=g, device=device) * std).to(torch.bfloat16).view(torch.int16)
        u = torch.rand(m, generator=g, device=device)
        sign = torch.randint(0, 2, (m,), generator=g, device=device, dtype=torch.int32)
        mant = torch.randint(1, 128, (m,), generator=g, device=device, dtype=torch.int32)
        sub = ((sign << 15) | mant).to(torch.int32)
        sub = torch.where(sub >= 32768, sub - 65536, sub).to(torch.int16)  # as signed 16-bit
        bits = torch.where(u < zero_frac, torch.zeros_like(gauss),
                           torch.where(u < zero_frac + subnormal_frac, sub, gauss))
        out[s:s + m] = bits.view(torch.bfloat16)
    return out


# ----------------------------------------------------------------- workloads

def workload(k: int, device="cpu", small: bool = False):
    """(data, calibration sample) of benchmark workload k (1, 2, 3 or 5).

    ``small=True`` draws a reduced instance of the same law (for CPU tests and
    oracle-sized parity cases): it spans many chunks and has a ragged tail.
    """
    if k == 1:
        rows = 257 if small else 8192
        x = rows_lognormal_scale(rows, 128, seed=DATA_SEED + 1, device=device)
        s = rows_lognormal_scale(512, 128, seed=CALIB_SEED + 1, device=device)
        return x.reshape(-1), s.reshape(-1)
    if k == 2:
        shape = (4, 2, 2, 33, 128) if small else KV_SHAPE
        x = kv_cache(shape, seed=DATA_SEED + 2, device=device)
        s = kv_cache_sample(1 << 16 if small else 1 << 20, device=device)
        return x.reshape(-1), s
    if k == 3:
        x = heavy_tailed((1 << 16) + 37 if small else 1 << 26, seed=DATA_SEED + 3, device=device)
        s = gaussian(1 << 16 if small else 1 << 20, seed=CALIB_SEED + 3, device=device)
        return x, s
    if k == 5:
        x = gradient_like((1 << 16) + 5 if small else 1 << 30, seed=DATA_SEED + 5, device=device)
        s = gradient_like(1 << 16 if small else 1 << 22, seed=CALIB_SEED + 5, device=device)
        return x, s
    raise ValueError(f"workload {k}: use sweep() for the message-size sweep (4)")


def workload_e5m2(device="cpu", small: bool = False):
    """(data, calibration sample) for the FP8 E5M2 codec: the KV-cache law of
    workload 2 quantised to E5M2 (round to nearest even, as an FP8 KV cache
    stores it), as uint8 bit patterns. The page measures FP8 KV from real
    models; this is its synthetic stand-in."""
    x, s = workload(2, device=device, small=small)
    return to_e5m2_bits(x), to_e5m2_bits(s)


def to_e5m2_bits(x: torch.Tensor) -> torch.Tensor:
    """E5M2 bit patterns (uint8) of x, rounded to nearest even."""
    return x.float().to(torch.float8_e5m2).view(torch.uint8)


def as_u8(x: torch.Tensor):
    """Host numpy uint8 copy of a one-byte tensor's bit patterns."""
    return x.detach().contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


def sweep_sample(device="cpu", n: int = 1 << 20) -> torch.Tensor:
    return gaussian(n, seed=CALIB_SEED + 4, device=device)


def sweep(nbytes: int, device="cpu", seed: int | None = None) -> torch.Tensor:
    """N(0, 1) buffer of ``nbytes`` raw BF16 bytes (message-size sweep)."""
    return gaussian(nbytes // 2, seed=(DATA_SEED + 4) if seed is None else seed, device=device)


def as_u16(x: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns."""
    import numpy as np
    return x.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
