"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each a replica with
its own timings; the whole-job figure uses the slowest rank's time and all
ranks' bytes, and both ranks agree on it."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as tmp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 0.5 * (rank + 1), 3.0 - rank]
        agg = bench.max_over_ranks(mine, world)
        v = bench.whole_job_gbs(1e9, world, agg[0])
        dist.barrier()
        q.put((rank, agg, v))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_whole_job_value():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, a0, v0), (r1, a1, v1) = res
    assert a0 == a1 == [2.0, 1.0, 3.0]
    assert v0 == v1 == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_reference_arm_rank_nonzero_does_no_work(capsys):
    import argparse
    import bench
    bench.run_reference(argparse.Namespace(steps=1, warmup=0, gpus=2), rank=1, world=2)
    assert capsys.readouterr().out == ""
