"""The benchmark's multi-rank path on CPU with two gloo ranks: the timing is
the max over ranks and the whole-job value counts every replica's work."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 15.0 and out[1] == 15.0


def test_whole_job_value_counts_replicas():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5  # no process group: identity
    one = bench.whole_job_tflops(133.9e12, 1, 100.0)
    assert abs(one - 1339.0) < 1e-9
    assert abs(bench.whole_job_tflops(133.9e12, 4, 100.0) - 4 * one) < 1e-9
