"""Multi-rank host logic of the benchmark on CPU with the gloo backend
(world size 2): the job time is the slowest rank's, the job rate counts every
rank's units (weak scaling, one replica per rank), and batch-row shards cover
the batch exactly once.  No GPU and no data-path collective are involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank * 0.25)  # rank 1 is slower
        r, w, local = bench.dist_env()
        q.put((rank, ms, r, w, local, bench.job_rate(w, 1000, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, r, w, local, rate in out:
        assert ms == pytest.approx(1.25)          # slowest rank
        assert (r, w, local) == (rank, 2, rank)
        assert rate == pytest.approx(2 * 1000 / 1.25e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_rate(1, 10, 2.0) == pytest.approx(5000.0)


@pytest.mark.parametrize("batch,world", [(8, 2), (8, 3), (5, 8), (32, 4), (1, 1)])
def test_shard_rows_cover_batch(batch, world):
    seen = []
    for r in range(world):
        lo, hi = bench.shard_rows(batch, r, world)
        assert 0 <= lo <= hi <= batch
        seen.extend(range(lo, hi))
    assert seen == list(range(batch))
