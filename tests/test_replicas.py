"""Multi-process bookkeeping of the throughput run, on CPU with the gloo backend (world size 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from folded_tensor_sequence_gb300.replicas import max_over_ranks, rank_env, whole_job_rate


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = rank_env()
        assert (env.world_size, env.rank, env.local_rank) == (world, rank, rank)
        dist.barrier()
        ms = max_over_ranks(times[rank])
        rate = whole_job_rate(env.world_size, 1000.0, 10, ms)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank_units():
    world, times = 2, [12.5, 40.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=10) for _ in range(world))
    for rank, ms, rate in got:
        assert ms == 40.0  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 * 10 / 0.040)  # both ranks' units over that time


def test_single_process_defaults():
    env = rank_env({})
    assert (env.world_size, env.rank, env.local_rank) == (1, 0, 0)
    assert max_over_ranks(3.25) == 3.25
    assert whole_job_rate(1, 64.0, 4, 2.0) == pytest.approx(64 * 4 / 0.002)
    with pytest.raises(ValueError):
        whole_job_rate(1, 1.0, 1, 0.0)
