"""The replica path of bench.py (N > 1 processes) on the CPU: two gloo ranks,
each with its own step times, agree on the slowest rank's times (the job's
pace), and the job throughput counts the rows of every rank.  The verify
step itself does not shard (replicas only), so this is all the data path
exchanges between ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, times, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        ms, e2e = bench.slowest_rank(times[rank][0], times[rank][1], dist, "cpu")
        q.put((rank, ms, e2e, bench.job_throughput(world, 16, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [(4.25, 4.375), (4.5, 4.125)]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r for r, *_ in res] == [0, 1]
    for _, ms, e2e, value in res:
        assert ms == 4.5 and e2e == 4.375  # each column's max over the ranks
        assert value == pytest.approx(2 * 16 / 4.5e-3)


def test_one_process_keeps_its_times():
    import bench
    assert bench.slowest_rank(4.25, 4.375, None, "cpu") == (4.25, 4.375)
    assert bench.job_throughput(1, 16, 4.0) == pytest.approx(4000.0)
