"""The bench's N > 1 path on CPU: two gloo ranks, each an independent replica of the workload.

Each rank plans the same workload (host only), the job time is the slowest rank's, and the
job throughput counts every rank's bytes. No data-path collective exists: replicas share
nothing but the barrier and the max-over-ranks timing reduction.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import dtensor_resharding_gb300 as R
        import synthetic as S
        wl = S.dense_ffn(layers=2, hidden=256, ffn=1000)
        st = R.reshard_plan_stats(R.plan_workload(wl))
        # rank r pretends its timed region took 10 + r ms
        ms = bench.max_over_ranks(10.0 + rank, world)
        dist.barrier()
        out[rank] = (st["bytes_written"], st["items"], ms,
                     bench.job_throughput(wl.dst_bytes(), 5, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][:2] == res[1][:2]              # identical replica plans
    assert res[0][2] == res[1][2] == 11.0         # both see the slowest rank's time
    assert res[0][3] == pytest.approx(world * res[0][0] * 5 / 11e-3 / 1e9)
