"""Multi-rank host logic on CPU with 2 gloo ranks (no GPU).

The path partitions by image with no exchange step: each rank runs its own
images.  These tests check bench.py's rank plumbing (image sharding, barrier,
max-over-ranks timing) and that splitting a batch's images over ranks, running
the oracle on each shard and gathering the results reproduces the unsharded
oracle bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from ragged_attention_token_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = W.make_custom(5, 23, 2, None, random_mask=True, seed=11)
        keep = case.keep.numpy()
        qn, kn, vn = (x.double().numpy() for x in (case.q, case.k, case.v))
        s0, s1 = bench.image_shard(case.B, rank, world)
        out, *_ = oracle.pipeline(keep[s0:s1], qn[s0:s1], kn[s0:s1], vn[s0:s1], 0.125)
        parts = [None] * world
        dist.all_gather_object(parts, (s0, s1, out))
        bench.barrier(world)
        slowest = bench.max_over_ranks(float(rank + 1), world, torch.device("cpu"))
        if rank == 0:
            full, *_ = oracle.pipeline(keep, qn, kn, vn, 0.125)
            merged = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=0)
            covered = sorted((p[0], p[1]) for p in parts)
            q.put((np.array_equal(merged, full), covered, slowest))
    finally:
        dist.destroy_process_group()


def test_image_shard_covers_batch():
    for B in (1, 2, 5, 64, 257):
        for world in (1, 2, 3, 8):
            ranges = [bench.image_shard(B, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [e - s for s, e in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_shard_images_and_time_max():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    equal, covered, slowest = q.get()
    assert equal
    assert covered == [(0, 3), (3, 5)]
    assert slowest == 2.0
