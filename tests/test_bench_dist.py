"""The benchmark's multi-rank path on the CPU: two gloo ranks, each timing its own
batch (no collective on the data path), combined as all ranks' queries over the
slowest rank's time."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    d = bench.Dist(backend="gloo")
    try:
        d.barrier()
        # rank r processed 64 * (r + 1) queries in (r + 1) * 0.5 seconds
        qps, slowest = bench.aggregate(d, 64.0 * (rank + 1), 0.5 * (rank + 1))
        queue.put((rank, qps, slowest))
    finally:
        d.close()


def test_two_rank_aggregation_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for _, qps, slowest in got:
        assert slowest == pytest.approx(1.0)
        assert qps == pytest.approx((64.0 + 128.0) / 1.0)


def test_single_process_needs_no_group():
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    assert bench.aggregate(d, 128.0, 0.25) == (512.0, 0.25)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
