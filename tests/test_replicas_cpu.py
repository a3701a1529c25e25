"""The multi-GPU path is replicas only: each rank runs the whole layer on its
own tokens, with no data exchange; bench.py's ranks meet at barriers and take
the slowest rank's time.  Exercised here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        # rank r took (r + 1) ms per step on its own 1000 tokens
        ms_max = d.max(float(rank + 1))
        q.put((rank, d.world, ms_max, bench.whole_job_rate(1000, d.world, ms_max)))
        d.barrier()
    finally:
        d.close()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, world, ms_max, rate in got:
        assert world == 2
        assert ms_max == 2.0                 # the slower rank's time, on every rank
        assert rate == pytest.approx(1000 * 2 / 2e-3)   # both replicas' tokens over that time


def test_single_process_needs_no_group():
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    assert d.max(3.5) == 3.5
    assert bench.whole_job_rate(32768, 1, 4.0) == pytest.approx(32768 / 4e-3)
