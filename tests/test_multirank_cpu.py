"""The N > 1 host logic of bench.py on CPU with the gloo backend (world size 2):
the barrier, the max-over-ranks of the timed interval, the weak-scaling value
(units of all ranks / the slowest rank's time), and the reference arm printing
from rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch

    import bench

    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    mine = 10.0 + 5.0 * rank  # rank 1 is the slower one
    got = bench.max_over_ranks(dist, mine, torch.device("cpu"))
    out.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_weak_scaling_value_uses_all_ranks_and_the_slowest_time():
    sys.path.insert(0, ROOT)
    import bench

    T, H, D = bench.T_TOKENS, bench.HEADS, bench.HEAD_DIM
    step = bench.scatter_bytes(T, H, D) + bench.restore_bytes(T, H, D, T // bench.BLOCK)
    assert step == 5_544_869_888 + 5_536_743_428
    # value = world * bytes / max-rank time
    ms = 2.0
    assert abs(2 * step / (ms * 1e-3) / 1e9 - 2 * step / 2e6) < 1e-6


def test_kernel_line_quantiles_by_nearest_rank():
    """P50 / P90 of the per-step kernel times: nearest rank on the sorted times."""
    sys.path.insert(0, ROOT)
    import bench

    assert bench.nearest_rank([5.0, 1.0, 3.0, 2.0, 4.0], 0.5) == 3.0
    assert bench.nearest_rank([5.0, 1.0, 3.0, 2.0, 4.0], 0.9) == 5.0
    assert bench.nearest_rank([float(i) for i in range(1, 101)], 0.9) == 90.0
    assert bench.nearest_rank([7.0], 0.9) == 7.0
    row = bench.kernel_row([1.0, 1.2, 0.8, 1.0], 6_000_000_000, 6000.0)
    assert row["ms"] == 1.0 and row["p50_ms"] == 1.0 and row["p90_ms"] == 1.2
    assert row["GB/s"] == 6000.0 and row["frac"] == 1.0


def test_reference_arm_prints_from_rank_zero_only():
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2")
    outs = []
    for rank in (1,):
        e = dict(env, RANK=str(rank), LOCAL_RANK=str(rank))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--gpus", "2", "--steps", "1", "--warmup", "0"],
                           env=e, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        outs.append(r.stdout.strip())
    assert outs == [""]


@pytest.mark.parametrize("steps", [1])
def test_reference_arm_json_line(steps):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", str(steps), "--warmup", "0", "--ref-seconds", "2"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
