"""The benchmark's multi-process host logic on CPU, world size 2 over gloo:
rank environment, the barrier, the max-over-ranks timing reduction and the
whole-job rate.  The data path shards by rows with no collective, so these are
the only cross-rank steps."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    ws, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    try:
        bench.barrier()
        t = bench.reduce_max(0.5 + rank)          # rank 1 is the slow one
        rate = bench.whole_job_rate(1000.0, ws, t)
        bench.barrier()
        out.put((r, ws, local, t, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
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
    assert [x[0] for x in res] == [0, 1]
    for r, ws, local, t, rate in res:
        assert ws == 2 and local == r
        assert t == 1.5                       # the max over ranks, seen by both
        assert rate == pytest.approx(1000.0 * 2 / 1.5)


def test_single_process_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench

    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_max(2.5) == 2.5       # no process group: identity
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
