"""The multi-process path of the benchmark on CPU (gloo, world size 2):
ranks are replicas, so the only cross-rank steps are the barrier, the max
of the ranks' times and the sum of their work; the reference arm runs on
rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    bench.barrier(ws)
    mx = bench.reduce_max(1.5 + rank, ws)
    rate = bench.job_rate(10.0 * (rank + 1), 2.0 + rank, ws)   # units, ms
    ref = bench.run_reference(None, ws, rank) if rank == 1 else "skipped"
    bench.barrier(ws)
    q.put((rank, mx, rate, ref))
    dist.destroy_process_group()


def test_two_gloo_ranks_sum_work_and_take_the_slowest_time():
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
    for rank, mx, rate, ref in out:
        assert mx == 2.5                                  # slowest rank's value
        assert rate == pytest.approx((10.0 + 20.0) / 3.0e-3)   # all units / slowest time
    assert out[1][3] is None                              # reference arm: rank 0 only


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.job_rate(6.0, 2.0, 1) == pytest.approx(3000.0)
