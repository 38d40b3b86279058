"""World-size-2 tests on CPU (gloo): the multi-process logic of the benchmark
and the det-train page's multi-rank claim, without any GPU.

The page (sections "Correctness" and "Real multi-GPU") sums K-sharded
partials across ranks with a single int64 all-reduce of the accumulator
digits, and reports the same result digest on every rank at world sizes 1
and 4.  Here each rank
computes the oracle's digits of its own K-shard, the digits are summed with a
gloo all-reduce, and the canonical digits, the rounded result and its digest
must equal the single-process ones on every rank.
"""
import hashlib
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _digest(arr):
    return hashlib.sha256(np.ascontiguousarray(arr).tobytes()).hexdigest()


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from exact_sum_gemm_gb300 import workloads as wl
        oracle.build()
        # benchmark helpers: the slowest rank's time, one seed per rank
        assert bench.max_over_ranks(10.0 + rank, dist, "cpu") == 10.0 + world - 1
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_seed(rank))
        assert len(set(seeds)) == world
        # K-sharded exact GEMM reduced across ranks with an int64 sum
        A = wl.normal_f32((24, 300), 5, 0)
        B = wl.loguniform_f32((20, 300), 5, 1, lo=-30, hi=30)
        k0, k1 = wl.kshard_cuts(300, world, seed=11)[rank]
        part = oracle.gemm_digits(A[:, k0:k1], B[:, k0:k1])
        t = torch.from_numpy(part.copy())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        summed = oracle.canonicalize(t.numpy())
        result = oracle.finalize(t.numpy())
        np.save(os.path.join(out_dir, f"digits{rank}.npy"), summed)
        np.save(os.path.join(out_dir, f"result{rank}.npy"), result)
    finally:
        dist.destroy_process_group()


def test_world_size_2_gloo(tmp_path, oracle_mod):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    from exact_sum_gemm_gb300 import workloads as wl
    A = wl.normal_f32((24, 300), 5, 0)
    B = wl.loguniform_f32((20, 300), 5, 1, lo=-30, hi=30)
    want_digits = oracle_mod.gemm_digits(A, B)
    want = oracle_mod.gemm(A, B)
    for r in range(world):
        np.testing.assert_array_equal(np.load(tmp_path / f"digits{r}.npy"), want_digits)
        got = np.load(tmp_path / f"result{r}.npy")
        np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
        assert _digest(got) == _digest(want)          # same digest at world size 1 and 2
