"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, barrier and
max-over-ranks of the timed region, and the whole-job throughput formula
(replicas: every rank processes the full workload)."""

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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(world)
    d.init("gloo")
    d.barrier()
    slowest = d.max(10.0 + rank)          # rank 1 is the slow one
    d.barrier()
    d.close()
    q.put((rank, slowest))


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: 11.0, 1: 11.0}


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput(1, 3 * 2**30, 10, 5.0)
    assert one == pytest.approx(3 * 2**30 * 10 / 5e-3 / 1e9)
    assert bench.job_throughput(4, 3 * 2**30, 10, 5.0) == pytest.approx(4 * one)


def test_dist_rejects_mismatched_world(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.Dist(4)


@pytest.mark.parametrize("op", ["residual_layernorm", "rmsnorm", "softmax"])
@pytest.mark.parametrize("threads", [1, 3, 8, 40])
def test_cpu_baseline_row_blocks_cover_every_row_once(op, threads):
    """The all-core CPU baseline splits rows into contiguous blocks; together
    they must equal one oracle call over all rows, bit for bit."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import synth
    rows, width = 37, 96
    x = synth.rows_of(3, rows, width, which="x")
    r = synth.rows_of(3, rows, width, which="r") if op == "residual_layernorm" else None
    orc = oracle.get()
    eps = oracle.kernel_eps(bench.EPS)
    parts = bench.oracle_rows(orc, op, x, r, eps, threads)
    assert len(parts) == min(threads, rows)
    assert np.array_equal(np.concatenate(parts), orc.run(op, x, r, eps))


def _bench(args, env_extra=None):
    import json
    import subprocess
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference`: the FP64 oracle on the host cores, one
    JSON line with the metric and unit our arm prints for the same workload
    (and the same config object), no GPU work."""
    sys.path.insert(0, ROOT)
    import bench
    out = _bench(["--impl", "reference", "--steps", "3", "--warmup", "3", "--rows", "2048",
                  "--width", "512"])
    assert len(out) == 1
    d = out[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s"
    assert d["metric"] == bench.metric_of("residual_layernorm", 2048, 512)
    assert bench.metric_of("residual_layernorm", 65536, 4096) == bench.METRIC
    assert d["config"] == bench.workload_config("residual_layernorm", 2048, 512, 1)
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["gpu_launches"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    out = _bench(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
                  "--rows", "256", "--width", "256"],
                 {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out == []
