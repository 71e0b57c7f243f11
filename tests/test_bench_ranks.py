"""The replica (N > 1) path of bench.py on CPU: two gloo ranks check the
barrier and the whole-job reduction (sum of bytes over the slowest rank's
time), with no GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r read (r + 1) GB in (10 + 5 r) ms
        gbs, ms, total = bench.whole_job_gbs((rank + 1) * 1e9, 10.0 + 5.0 * rank, world)
        results[rank] = (gbs, ms, total, bench.max_over_ranks(float(rank), world),
                         bench.sum_over_ranks(1.0, world))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_whole_job_numbers():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    for r in range(world):
        gbs, ms, total, mx, sm = res[r]
        assert ms == pytest.approx(15.0)             # slowest rank's time
        assert total == pytest.approx(3e9)           # all ranks' bytes
        assert gbs == pytest.approx(3e9 / 15e-3 / 1e9)
        assert mx == 1.0 and sm == 2.0
