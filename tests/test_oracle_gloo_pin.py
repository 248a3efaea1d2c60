"""Pin the oracle against an independent allreduce: torch.distributed (gloo).

Several processes, one per rank, each hold one rank's vector and call
``dist.all_reduce(SUM)``; gloo's own algorithm and summation order differ
from the ring's, so the inputs are small integers, for which every order is
exact.  The oracle's result on the same vectors must then be identical, and
DDP's average (divide by world size, "DDP 与 Ring All-Reduce：梯度同步不是
一次 AllReduce 就完事" section 05; "Day 17 · 梯度的集体行动" Reducer
pseudo-code) must equal gloo's sum divided by the world size.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = workloads.small_int_f32(n, seed=rank)
        dist.all_reduce(x, op=dist.ReduceOp.SUM)
        np.save(os.path.join(out_dir, f"r{rank}.npy"), x.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n", [(2, 37), (3, 64)])
def test_oracle_matches_gloo_allreduce_on_exact_inputs(tmp_path, world, n):
    mp.start_processes(_worker, args=(world, _free_port(), n, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    gloo = [np.load(tmp_path / f"r{r}.npy") for r in range(world)]
    x = workloads.rank_vectors(world, n, kind="int").numpy()
    summed = oracle.ring_allreduce_2d(x.copy(), oracle.F32, divisor=0)
    averaged = oracle.ring_allreduce_2d(x.copy(), oracle.F32, divisor=world)
    for r in range(world):
        np.testing.assert_array_equal(summed[r], gloo[r])
        np.testing.assert_array_equal(averaged[r], (gloo[r].astype(np.float64) / world).astype(np.float32))
