"""Multi-rank bench logic on CPU: world_size 2 over gloo (the GPU run uses NCCL).

Each rank runs an independent replica; the job time is the slowest rank's and
the throughput counts every rank's rows.  The reference arm prints only on
rank 0.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.5, 30.0][rank]
    mx = bench.max_over_ranks(local_ms)
    gbs = bench.job_throughput_gbs(1_000_000, 10, world, mx)
    dist.barrier()
    q.put((rank, mx, gbs))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, gbs in res:
        assert mx == 30.0
        assert gbs == pytest.approx(1_000_000 * 10 * 2 / 0.030 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.job_throughput_gbs(2e9, 1, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_silent_on_other_ranks(capsys):
    class A:
        config, warmup, steps, ref_rows = "tiny", 3, 1, 4
    bench.run_reference(A, rank=1, world=2)
    assert capsys.readouterr().out == ""
