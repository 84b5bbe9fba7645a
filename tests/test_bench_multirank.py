"""The bench's multi-rank host logic with two gloo ranks on CPU: max over ranks and the barrier.

Every rank runs its own replica of the workload (no data-path collective), so the only
cross-rank steps are the barrier around the timed region and the max of the timings.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        got = bench.max_over_ranks(10.0 + 7.0 * rank, w)
        bench.barrier(w)
        q.put((rank, w, r, local, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r[0], r[1], r[2], r[3]) for r in res] == [(0, 2, 0, 0), (1, 2, 1, 1)]
    assert all(r[4] == 17.0 for r in res)


def test_single_rank_helpers_are_identity(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
