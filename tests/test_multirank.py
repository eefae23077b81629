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


def _slab_worker(rank, world, port, q):
    """One rank of a batch-split run on CPU: it scans its batch rows with the
    oracle; rank 0 gathers the slabs with gloo."""
    import numpy as np
    import torch
    import torch.distributed as dist
    from oracle import ref_scan
    from selective_state_space_fwd_gb300 import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.WORKLOADS[4].scaled(batch=5, seqlen=300, dim=24)
        inp = W.make_inputs(w)
        lo, hi = bench.shard_rows(w.batch, rank, world)
        mine = bench.slice_rows(inp, lo, hi)
        y, s = ref_scan.scan_fwd(mine["x"], mine["delta"], mine["A"], mine["B"], mine["C"],
                                 mine["D"], mine["z"], mine["valid_len"],
                                 chunk_len=w.chunk_len, threads=1)
        # gather variable-sized slabs: pad to the largest shard
        per = -(-w.batch // world)
        pad_y = np.zeros((per,) + y.shape[1:])
        pad_s = np.zeros((per,) + s.shape[1:])
        pad_y[:hi - lo], pad_s[:hi - lo] = y, s
        ys = [torch.zeros(pad_y.shape, dtype=torch.float64) for _ in range(world)]
        ss = [torch.zeros(pad_s.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(ys, torch.from_numpy(pad_y))
        dist.all_gather(ss, torch.from_numpy(pad_s))
        if rank == 0:
            parts = [bench.shard_rows(w.batch, r, world) for r in range(world)]
            y_all = np.concatenate([ys[r].numpy()[:h - l] for r, (l, h) in enumerate(parts)])
            s_all = np.concatenate([ss[r].numpy()[:h - l] for r, (l, h) in enumerate(parts)])
            y1, s1 = ref_scan.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                       inp["D"], inp["z"], inp["valid_len"],
                                       chunk_len=w.chunk_len, threads=1)
            q.put((bool(np.array_equal(y_all, y1)), bool(np.array_equal(s_all, s1))))
    finally:
        dist.destroy_process_group()


def test_batch_split_slabs_reassemble_the_single_rank_result():
    """Splitting one workload's batch rows across two ranks (bench.py
    --split-batch) needs no exchange: the slabs each rank computes, put back in
    row order, are the single-rank result bit for bit."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_slab_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    same_y, same_s = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert same_y and same_s
