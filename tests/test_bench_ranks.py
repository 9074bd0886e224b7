"""The multi-rank host logic of bench.py, on CPU: two gloo ranks on 127.0.0.1.

With N > 1 every rank runs one replica of the workload; the job's time is the
slowest rank's (max over ranks) and its rate counts the units of all ranks."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [12.5, 20.0][rank]  # this rank's timed milliseconds
    got = bench.max_over_ranks(mine, world, device="cpu")
    rate = bench.whole_job_rate(10, world, got)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, rate))


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]  # both ranks see the slowest time
    assert all(abs(r[2] - 2 * 10 / 0.020) < 1e-9 for r in res)  # 20 units in 20 ms


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_rate(50, 1, 25.0) == 2000.0
