"""Bounded waits of the TMA-staged kernels, made to run out on purpose.

A collective waits for every rank, so a rank that never joins a step stalls
the others without an error ("Day 17 · 梯度的集体行动", "INVARIANT 2" and
"常见疑问" Q2).  On one GPU the "ranks" are copies that a producer warp stages
into shared memory; ddp_plant_stall makes that producer stop issuing them at
one tile, so the consumer warps wait for data that never arrives.  The wait
limit (ddp_set_wait_limit_ms, here 100 ms) must end that wait: the call
returns, the device status word reads DDP_ERR_TIMEOUT, and the context stays
usable -- the next clean call gives the oracle's bits again.

Nothing here faults or hangs a GPU: the planted producer issues no copy at
all for the stalled tile (nothing is left in flight, nothing is out of
bounds), and every wait has its limit.
"""
import time

import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import workloads
from gpu_util import assert_bits_equal, f32_or_bits, oracle_allreduce

pytestmark = pytest.mark.gpu
TIMEOUT = -4


def _limited(ms):
    class Ctx:
        def __enter__(self):
            self.prev = ddp.ddp_set_wait_limit_ms(ms)
            self.prev_kernel = ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_TMA)
            ddp.ddp_device_status(clear=True)

        def __exit__(self, *exc):
            ddp.ddp_plant_stall(-1)
            ddp.ddp_set_fused_kernel(self.prev_kernel)
            ddp.ddp_set_wait_limit_ms(self.prev)
    return Ctx()


@pytest.mark.parametrize("tile", [0, 500, 1023])
def test_fused_tma_wait_runs_out_on_a_planted_stall(tile):
    # N = 8 x 2^21 fp32: chunks of 1 MiB, tiles of 8 KB, 1024 tiles over the
    # persistent grid; the stalled tile is the CTA's first, a middle one, or
    # the last one of the launch
    N, S = 8, 1 << 21
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, seed0=21)
    want = oracle_allreduce(x.numpy(), N)
    with _limited(100):
        xd = x.cuda()
        torch.cuda.synchronize()
        ddp.ddp_plant_stall(tile)
        t0 = time.perf_counter()
        ddp.ring_allreduce_fused(xd, N)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert ddp.ddp_device_status(clear=True) == TIMEOUT
        assert 0.09 <= dt < 1.5, dt
        # the stalled CTA stopped: its chunk is left unreduced somewhere
        assert not np.array_equal(f32_or_bits(xd).view(np.uint32), want.view(np.uint32))
        # the context is still good: a clean call gives the oracle's bits
        xd = x.cuda()
        ddp.ring_allreduce_fused(xd, N)
        torch.cuda.synchronize()
        assert ddp.ddp_device_status(clear=True) == 0
        assert_bits_equal(f32_or_bits(xd), want, f"clean call after stall at tile {tile}")


def test_view_tma_wait_runs_out_on_a_planted_stall():
    # one bucket of two 2^20-element members per rank, every body aligned,
    # 8 MiB over all ranks: the TMA view kernel takes it
    N, n = 8, 1 << 20
    flat = workloads.rank_vectors(N, 2 * n, "randn", std=1e-2, seed0=31)
    want = oracle_allreduce(flat.numpy(), N)
    with _limited(100):
        g = flat.cuda()
        grads = [[g[r, :n], g[r, n:]] for r in range(N)]
        torch.cuda.synchronize()
        ddp.ddp_plant_stall(10)
        t0 = time.perf_counter()
        ddp.ddp_bucket_allreduce_view(grads, [0, n], 2 * n, N)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert ddp.ddp_device_status(clear=True) == TIMEOUT
        assert 0.09 <= dt < 1.5, dt
        g = flat.cuda()
        grads = [[g[r, :n], g[r, n:]] for r in range(N)]
        ddp.ddp_bucket_allreduce_view(grads, [0, n], 2 * n, N)
        torch.cuda.synchronize()
        assert ddp.ddp_device_status(clear=True) == 0
        assert_bits_equal(f32_or_bits(g), want, "view: clean call after a stall")


def test_plant_beyond_the_launch_stalls_nothing():
    # a tile number past the launch's last tile plants nothing, and the
    # launch takes (clears) the plant: neither call times out
    N, S = 8, 1 << 21
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, seed0=41)
    want = oracle_allreduce(x.numpy(), N)
    with _limited(100):
        for _ in range(2):
            xd = x.cuda()
            ddp.ddp_plant_stall(1 << 40)
            ddp.ring_allreduce_fused(xd, N)
            torch.cuda.synchronize()
            assert ddp.ddp_device_status(clear=True) == 0
            assert_bits_equal(f32_or_bits(xd), want, "plant beyond the launch")
