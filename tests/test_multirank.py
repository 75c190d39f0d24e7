"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2).

On one box the merge has no exchange step, so under torchrun each rank merges
its own replica; what crosses ranks is only the timing: the whole-job figure is
every rank's bytes over the slowest rank's time, and the reference arm runs on
rank 0 alone."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        elapsed = [2.0, 3.0][rank]
        agg = bench.aggregate(per_rank_bytes=1_000_000_000, steps=4, elapsed_s=elapsed, ws=ws)
        bench.barrier(ws)
        ref_rc = None
        if rank == 1:
            args = bench.parse(["--impl", "reference"])
            from checkpoint_averaging_gb300 import workloads as W
            ref_rc = bench.run_reference(args, W.workload("pythia14m"), ws, rank)
        q.put((rank, agg, bench.dist_env(), ref_rc))
    finally:
        dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_and_counts_all_bytes():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(ws):
        rank, agg, env, ref_rc = q.get(timeout=120)
        results[rank] = (agg, env, ref_rc)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (agg, env, ref_rc) in results.items():
        assert env == (2, rank, rank)
        assert agg["seconds"] == pytest.approx(3.0)
        assert agg["gbs"] == pytest.approx(2 * 4 * 1.0 / 3.0)
        assert agg["ms_per_step"] == pytest.approx(750.0)
    assert results[1][2] == 0  # rank 1 leaves the reference arm without work


def test_single_rank_aggregate():
    import bench
    agg = bench.aggregate(per_rank_bytes=10 ** 9, steps=2, elapsed_s=0.5, ws=1)
    assert agg["gbs"] == pytest.approx(4.0)
