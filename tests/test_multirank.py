"""The benchmark's multi-rank logic (replicas only: no data-path collective) on
CPU with the gloo backend, world size 2: every rank times its own replica, the
job time is the slowest rank's, and the job throughput counts all replicas.
The reference arm runs on rank 0 only; other ranks exit without work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 20.0][rank]                     # rank 1 is the slow replica
    got = bench.max_over_ranks(ms, world, device="cpu")
    value = bench.job_throughput(1e9, 10, world, got)
    dist.barrier()
    q.put((rank, got, value))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    os.environ["PYTHONPATH"] = root + os.pathsep + os.environ.get("PYTHONPATH", "")
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
    for rank, ms, value in res:
        assert ms == 20.0                        # both ranks agree on the slowest time
        assert value == pytest.approx(2 * 1e9 * 10 / 0.020 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(1e9, 2, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_is_rank0_only():
    import argparse
    import bench
    args = argparse.Namespace(workload="gpt2_c_attn_1tok", ne11=0, steps=1, warmup=1)
    assert bench.run_reference(args, rank=1, world=2) is None
