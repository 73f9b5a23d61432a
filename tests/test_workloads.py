"""The synthetic inputs follow the recipe the benchmark and the parity tests
state for them (seeded, so every run sees the same tensors): row scales
log-uniform in [0.05, 4]; a KV cache whose K and V share one scale per
(layer, head), with 0.1 % of channels amplified x20; a heavy-tailed law that
puts a few percent of values outside an N(0,1) codebook; a gradient-like
buffer with 10 % exact zeros and 1 % subnormals."""
import math

import numpy as np
import torch

import lossless_bf16_exponent_gb300.workloads as W


def test_seeded_and_deterministic():
    a = W.gaussian(4096, seed=1)
    assert torch.equal(a.view(torch.int16), W.gaussian(4096, seed=1).view(torch.int16))
    assert not torch.equal(a.view(torch.int16), W.gaussian(4096, seed=2).view(torch.int16))


def test_row_scales_log_uniform():
    x = W.rows_lognormal_scale(rows=2048, cols=128, seed=7).float()
    s = x.std(dim=1)
    assert x.shape == (2048, 128)
    assert 0.04 < s.min() and s.max() < 4.6
    # log-uniform: log-scales spread evenly over [log 0.05, log 4]
    ls = torch.log(s)
    lo, hi = math.log(0.05), math.log(4.0)
    frac_low_half = ((ls < (lo + hi) / 2).float().mean()).item()
    assert 0.42 < frac_low_half < 0.58


def test_kv_cache_scales_and_outlier_channels():
    shape = (8, 2, 4, 256, 128)  # 8192 channels -> 8 outlier channels
    x = W.kv_cache(shape, seed=3).float()
    std = x.std(dim=3)  # [L, KV, H, D]: per channel over tokens
    head = std.median(dim=3).values  # [L, KV, H]
    # K and V of one (layer, head) share the scale
    ratio = head[:, 0] / head[:, 1]
    assert torch.all((ratio > 0.85) & (ratio < 1.15))
    assert head.min() > 0.08 and head.max() < 9.0
    # outliers: channels about 20x their head's typical channel
    rel = std / head.unsqueeze(-1)
    n_out = int((rel > 8).sum())
    assert n_out == round(0.001 * 8 * 2 * 4 * 128)
    assert float(rel[rel > 8].min()) > 15 and float(rel[rel > 8].max()) < 25


def test_heavy_tailed_escapes_an_n01_codebook(orc):
    x = W.heavy_tailed((1 << 18) + 3, seed=11)
    s = W.gaussian(1 << 16, seed=12)
    exps = orc.calibrate(W.as_u16(s))
    rc, stream = orc.encode(W.as_u16(x), exps, 1024)
    assert rc == 0
    m = int(np.frombuffer(stream[24:32].tobytes(), dtype="<u8")[0])
    assert 0.01 < m / x.numel() < 0.08


def test_gradient_like_zeros_and_subnormals():
    n = 1 << 20
    x = W.gradient_like(n, seed=5)
    u = W.as_u16(x)
    zeros = np.count_nonzero(u == 0)
    e = (u >> 7) & 0xFF
    sub = np.count_nonzero((e == 0) & ((u & 0x7F) != 0))
    assert abs(zeros / n - 0.10) < 0.005
    assert abs(sub / n - 0.01) < 0.002
    rest = x.float()[torch.from_numpy(e.astype(np.int64) != 0)]
    assert abs(rest.std().item() - 1e-3) < 5e-5
