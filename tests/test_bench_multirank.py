"""The benchmark's multi-rank logic on CPU (two gloo ranks, no GPU).

Each rank owns an independent problem (weak scaling, no data-path
collective); the only cross-rank steps are the barriers around the timed
region and the max over ranks of the step time.  Whole-job throughput is the
units of all ranks divided by the slowest rank's time, and the reference arm
prints from rank 0 only.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _aggregate_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    # rank r took (r + 1) seconds for 100 units
    value, t = bench.aggregate(100.0, float(rank + 1), world)
    mx = bench.max_over_ranks(10.0 * (world - rank), world)
    bench.barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, value, t, mx))


def test_aggregate_takes_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_aggregate_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, t, mx in out:
        assert t == 2.0                       # the slowest rank's seconds
        assert value == pytest.approx(100.0 * world / 2.0)
        assert mx == 20.0


def test_single_rank_aggregate_is_local():
    assert bench.aggregate(50.0, 2.0, 1) == (25.0, 2.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def _reference_worker(rank, world, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "parity_m1_k256_n64", "--steps", "3",
                         "--warmup", "3"])
    q.put((rank, rc, buf.getvalue()))


def test_reference_arm_prints_on_rank0_only():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reference_worker, args=(r, world, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rc0, text0), (r1, rc1, text1) = out
    assert rc0 == 0 and rc1 == 0
    assert text1 == ""
    line = json.loads(text0.strip())
    assert line["impl"] == "reference"
    assert line["n_gpus"] == world and line["scaling"] == "weak"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["value"] > 0
