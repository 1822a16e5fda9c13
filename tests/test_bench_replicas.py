"""The multi-GPU path of bench.py runs independent replicas (one per rank,
no data exchange); the only collective is the max of the timed region.  Checked
with two gloo ranks on CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [12.0, 20.0][rank]                    # rank 1 is the slow one
    job = bench.job_time_ms(local, world, "cpu")
    value = bench.job_tokens_per_s(2048, 10, world, job)
    q.put((rank, job, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, job, value in res:
        assert job == pytest.approx(20.0)
        assert value == pytest.approx(2048 * 10 * 2 / 20e-3)


def test_single_rank_is_local_time():
    import bench
    assert bench.job_time_ms(7.5, 1) == 7.5
    assert bench.job_tokens_per_s(16, 4, 1, 2.0) == pytest.approx(16 * 4 / 2e-3)
