"""The benchmark's JSON line carries every key of its contract, with the
whole-step value, per-op means and medians, the roofline of the slower op and
its fraction of the peak; checked on the CPU with made-up timings."""
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
        "median_us"}


def _line(enc_ms, dec_ms):
    n = 268435456
    raw = 2 * n
    nbytes = 404_590_401
    args = types.SimpleNamespace(steps=10, warmup=3, tokens=2048)
    med = {"calibrate": 9.5, "encode": 162.7, "decode": 149.2}
    return bench.report(args, 1, 0, n, raw, nbytes, 296_000, max_ms=10 * (enc_ms + dec_ms + 0.01),
                        total_raw=10 * raw, cal_ms=0.01, enc_ms=enc_ms, dec_ms=dec_ms, e2e=None, cpu=None,
                        clocks={}, sample=None, median_us=med), raw, nbytes


def test_report_has_every_contract_key():
    line, raw, nbytes = _line(0.1632, 0.1497)
    assert KEYS <= set(line)
    json.dumps(line)  # one JSON line
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["higher_is_better"] is True
    assert line["gpu_launches"] == bench.KERNELS_PER_STEP * 10
    assert line["median_us"]["encode"] == 162.7 and line["encode_us"] == 163.2
    step_s = (0.1632 + 0.1497 + 0.01) * 1e-3
    assert abs(line["value"] - raw / step_s / 1e9) < 0.01


def test_roofline_is_the_slower_op():
    for enc_ms, dec_ms, kernel in ((0.1632, 0.1497, "encode"), (0.14, 0.15, "decode")):
        line, raw, nbytes = _line(enc_ms, dec_ms)
        r = line["roofline"]
        assert r["kernel"] == kernel and r["bound"] == "hbm" and r["unit"] == "GB/s"
        ms = enc_ms if kernel == "encode" else dec_ms
        assert abs(r["achieved"] - (raw + nbytes) / (ms * 1e-3) / 1e9) < 0.1
        assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3


def test_chunk_slices_cover_the_input_at_chunk_boundaries():
    for n, parts in ((1, 4), (1024, 16), (3 * 1024 + 5, 2), (268435456, 16), (1000003, 72)):
        sl = bench.chunk_slices(n, parts)
        assert sl[0][0] == 0 and sl[-1][1] == n and len(sl) <= parts
        for (a, b), (c, d) in zip(sl, sl[1:]):
            assert b == c and a % bench.CHUNK == 0 and c % bench.CHUNK == 0 and a < b


def test_chunk_parallel_oracle_round_trips():
    """The all-cores CPU baseline runs the unchanged oracle on chunk-aligned
    slices in threads; the slices decode back to the input."""
    import numpy as np

    import oracle

    o = oracle.Oracle()
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50_000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    exps = o.calibrate(x[:4096])
    ys = bench.oracle_parallel(o, x, exps, 4)
    assert len(ys) == 4 and np.array_equal(np.concatenate(ys), x)
