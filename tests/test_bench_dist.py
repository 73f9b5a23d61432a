"""The replica path of bench.py on CPU: two gloo ranks (127.0.0.1) check the
max-over-ranks time and the whole-job sum the JSON line is built from, and
that only rank 0 reports."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    ws, r = bench.init_dist("gloo")
    bench.barrier()
    t = 10.0 + 5.0 * rank           # per-rank elapsed ms
    units = 1000 * (rank + 1)       # per-rank processed bytes
    q.put((rank, ws, bench.max_over_ranks(t), bench.sum_over_ranks(units), bench.dist_env()))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_bench():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, tmax, usum, env in out:
        assert ws == 2
        assert tmax == 15.0          # the slowest rank sets the time
        assert usum == 3000.0        # whole-job units
        assert env == (2, rank, rank)


def test_single_process_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.sum_over_ranks(7) == 7.0
    bench.barrier()  # no process group: a no-op


def test_reference_line_shape(monkeypatch):
    """The reference arm's JSON keys, on a tiny slice (CPU only)."""
    sys.path.insert(0, ROOT)
    import bench
    import lossless_bf16_exponent_gb300.workloads as W

    tiny = W.workload(2, small=True)
    monkeypatch.setattr(W, "workload", lambda k, device="cpu", small=False: tiny)
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = bench.argparse.Namespace(steps=3, warmup=3)
    line = bench.run_reference(args)
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_threads()
    # the tiny workload fits in a step: the line says it ran the whole of it
    assert "whole workload" in line["config"]["step"] and "whole workload" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    for k in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "dtype",
              "data", "config"):
        assert k in line


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_only_rank0_reports(monkeypatch, rank):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", str(rank))
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.argparse.Namespace(steps=3, warmup=3)) is None
