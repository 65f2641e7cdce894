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


def test_attention_work_counts_visible_pairs():
    import bench

    # brute force: every (row, key) pair with key <= pos0 + row, two products of
    # d multiply-adds each per head
    T, pos0, nh, nkv, d = 5, 3, 4, 2, 8
    pairs = sum(1 for t in range(T) for j in range(pos0 + T) if j <= pos0 + t)
    flop, byts = bench.attention_work(T, pos0, nh, nkv, d)
    assert flop == 2 * 2 * d * nh * pairs
    assert byts == 4 * (T * nh * d * 2 + (pos0 + T) * nkv * d * 2)
    # the 9B chunk of 2048 rows: 34.4 GFLOP against 83.9 MB
    flop, byts = bench.attention_work(2048, 0, 16, 4)
    assert round(flop / 1e9, 1) == 34.4 and round(byts / 1e6, 1) == 83.9
