"""The benchmark's multi-rank logic on CPU with the gloo backend, world size 2.

Both parts of the path shard with no exchange step (layers or tokens for the
insert, chunks for the pack), so a multi-GPU run is independent shards: the only
collective is the max of the ranks' step times, and the job's throughput is the
bytes every rank moved over the slowest rank's time.  Under torchrun only rank
0 prints, and the reference arm does no work on other ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [0.5, 0.8][rank]  # rank 1 is the slow one
    m = bench.max_over_ranks(ms, world)
    v = bench.job_throughput(1e9, world, m)
    results[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_world2():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0] == res[1]
    m, v = res[0]
    assert m == 0.8
    assert abs(v - 2 * 1e9 / 0.8e-3 / 1e9) < 1e-9


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_throughput(2e9, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_does_nothing_on_other_ranks(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 3, 3, 2
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
