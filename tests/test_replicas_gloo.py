"""Host logic of the multi-GPU bench on CPU (gloo, world size 2).

Projections over independent problems shard without any exchange, so N GPUs
run N replicas: the bench takes the slowest rank's time and counts the work
of every rank. This checks that reduction with two gloo ranks.
"""

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


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t, u = bench.reduce_over_ranks(elapsed_s=1.0 + rank, units=10.0 * (rank + 1), world=world)
    bench.barrier(world)
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_two_rank_reduction():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == (2.0, 30.0) and out[1] == (2.0, 30.0)


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_over_ranks(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_runs_on_cpu(capsys):
    import json

    import bench

    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
