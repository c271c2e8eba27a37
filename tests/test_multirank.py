"""The multi-rank path of bench.py on CPU ranks (gloo, world size 2): the
path partitions into independent (batch, head) sequences, so ranks only agree
on the step time (the slowest rank's) and never exchange data; each rank
draws a different copy of the workload."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from selective_state_space_131_b300 import inputs
        ms_local = 1.0 + 0.5 * rank                      # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, world)
        rate = bench.whole_job_rate(4096, world, ms)
        shape = inputs.ScanShape(batch=1, seqlen=8, heads=2, headdim=4, dstate=4, rank=1, chunk=16, dtype="f32")
        x = inputs.make_scan_inputs(shape, bench.rank_seed(2, rank))["x"]
        gathered = [torch.empty_like(x) for _ in range(world)]
        dist.all_gather(gathered, x)
        out[rank] = (ms, rate, bool(torch.equal(gathered[0], gathered[1])))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_agree_on_the_slowest_step():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        ms, rate, same = res[rank]
        assert ms == pytest.approx(1.5)                       # the max over ranks
        assert rate == pytest.approx(2 * 4096 / 1.5e-3)      # whole job: both ranks' units
        assert not same                                        # distinct inputs per rank


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.whole_job_rate(100, 1, 2.0) == pytest.approx(5e4)
