"""GPU parity of the tree allreduce kernels against the oracle's binomial tree.

tree_allreduce_fused and tree_allreduce_staged, through the C ABI, bit-exact
against oracle.tree_allreduce on the same seeded inputs: every N in 1..9 with
every S in 0..70, larger N (fused up to 64, staged beyond), ragged multi-tile
sizes, buffers that are not 16-byte aligned, and an 8 x 1 GiB bucket
compared in full.
"""
import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import (assert_bits_equal, assert_canaries, assert_device_equals_host, f32_or_bits, from_np,
                      guarded_copy, host_snapshot, require_host_memory, run_rank_buffers)

pytestmark = pytest.mark.gpu

TREE = {"fused": ddp.tree_allreduce_fused, "staged": ddp.tree_allreduce_staged}


def oracle_tree(x, divisor):
    y = np.ascontiguousarray(x).copy()
    oracle.tree_allreduce_2d(y, oracle.BF16 if y.dtype == np.uint16 else oracle.F32, divisor)
    return y


def run(kernel, xh, divisor):
    storage, x = guarded_copy(from_np(xh))
    TREE[kernel](x, divisor)
    torch.cuda.synchronize()
    assert_canaries(storage, f"tree {kernel} {tuple(x.shape)}")
    return f32_or_bits(x)


@pytest.mark.parametrize("kernel", ["fused", "staged"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_exhaustive_small(kernel, dtype):
    for N in range(1, 10):
        for S in range(0, 71):
            xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", dtype=dtype, seed0=N * 77 + S))
            for div in (0, N):
                assert_bits_equal(run(kernel, xh, div), oracle_tree(xh, div), f"tree {kernel} N={N} S={S}")


@pytest.mark.parametrize("kernel,N", [("fused", 16), ("fused", 17), ("fused", 33), ("fused", 48), ("fused", 49),
                                      ("fused", 64), ("staged", 64), ("staged", 100)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_many_ranks(kernel, N, dtype):
    xh = f32_or_bits(workloads.rank_vectors(N, 1029, "randn", std=1e-2, dtype=dtype, seed0=N))
    assert_bits_equal(run(kernel, xh, N), oracle_tree(xh, N), f"tree {kernel} N={N}")


@pytest.mark.parametrize("kernel", ["fused", "staged"])
@pytest.mark.parametrize("N,S", [(3, 1_000_003), (8, (1 << 20) + 5), (5, 777_777)])
def test_many_tiles_ragged(kernel, N, S):
    for dtype in ("f32", "bf16"):
        xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=1))
        assert_bits_equal(run(kernel, xh, N), oracle_tree(xh, N), f"tree {kernel} N={N} S={S} {dtype}")


@pytest.mark.parametrize("kernel", ["fused", "staged"])
def test_unaligned(kernel):
    N, S = 6, 5000
    x = workloads.rank_vectors(N, S, "randn", seed0=2)
    store = torch.zeros((N, S + 8), device="cuda")
    rows = [store[r, 3:3 + S] for r in range(N)]
    for r in range(N):
        rows[r].copy_(x[r].cuda())
    TREE[kernel](rows, N)
    torch.cuda.synchronize()
    assert_bits_equal(np.stack([f32_or_bits(r) for r in rows]), oracle_tree(x.numpy(), N), f"unaligned {kernel}")


_gib = {}


@pytest.fixture(scope="module", autouse=True)
def _release_full_size_buffers():
    yield
    _gib.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["fused", "fused_vector", "staged"])
def test_one_gib_buckets_full(kernel):
    # 8 x 1 GiB fp32, every element of every rank against the oracle's tree
    N, S = 8, 1 << 28
    if not _gib:
        require_host_memory(N * S * 4, "8 x 1 GiB tree")
        x0 = torch.empty((N, S), device="cuda")
        for r in range(N):
            x0[r].copy_(workloads.randn_f32(S, r, 1e-2, device="cuda"))
        want = host_snapshot(x0)
        oracle.tree_allreduce_2d(want, oracle.F32, N)
        _gib["case"] = (x0, want)
    x0, want = _gib["case"]
    storage, x = guarded_copy(x0)
    if kernel == "fused_vector":                  # the size rule picks the TMA kernel here
        prev = ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_VECTOR)
        try:
            ddp.tree_allreduce_fused(x, N)
        finally:
            ddp.ddp_set_fused_kernel(prev)
    else:
        TREE[kernel](x, N)
    torch.cuda.synchronize()
    assert_canaries(storage, f"1 GiB tree {kernel}")
    assert_device_equals_host(x, want, f"1 GiB tree {kernel}")
    del x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_both_kernels_around_the_size_switch(dtype):
    # small buckets take the lane-group kernel, larger ones one thread per
    # vector; sizes on both sides of the switches (64, 128 and 512 KiB per
    # rank) with ragged tails, every lane split (P = 2 .. 32 lanes per
    # vector, one or two vectors per lane); then each kernel forced
    es = 2 if dtype == "bf16" else 4
    for N in (2, 3, 5, 8, 16, 17, 31, 33, 64):
        for kib in ((16, 64, 128, 512) if N <= 8 else (16, 64, 128)):
            for delta in (-3, 0, 5):
                S = kib * 1024 // es + delta
                xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=N + kib + delta))
                for div in (N, 3):
                    assert_bits_equal(run("fused", xh, div), oracle_tree(xh, div), f"tree N={N} S={S} div={div}")

    for kind in (ddp.DDP_FUSED_GROUP, ddp.DDP_FUSED_VECTOR, ddp.DDP_FUSED_TMA):
        # the last four sizes have whole 16-byte rows, which the TMA kernel
        # takes (tiles over the whole bucket; 16 and 64 ranks: both of its
        # rank-table sizes); the first three make a forced TMA fall back
        for N, S in ((2, 3 * 1024 * 1024 // es + 7), (7, 99_999), (64, 40_000 + 3), (2, 1 << 20),
                     (8, 3 * 1024 * 1024 // es), (16, 123_456), (64, 40_000)):
            xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=N + kind))
            prev = ddp.ddp_set_fused_kernel(kind)
            try:
                got = run("fused", xh, N)
            finally:
                ddp.ddp_set_fused_kernel(prev)
            assert_bits_equal(got, oracle_tree(xh, N), f"tree forced kernel {kind} N={N} S={S}")


# Buckets of at least 128 MiB over all ranks run the vector tree with one block
# per tile of vectors, the elements past the last whole vector on block 0; a
# CTA cap makes the launch loop over the tiles.  Separate aligned rank buffers
# with ragged lengths, compared in full.
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,S", [(2, 16_777_219), (5, 6_710_891), (8, 4_194_307), (16, 2_097_155),
                                 (33, 1_016_809)])
def test_vector_tree_one_block_per_tile(dtype, N, S):
    S = S * 2 if dtype == "bf16" else S
    assert N * S * (2 if dtype == "bf16" else 4) >= 128 << 20
    xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=7 * N))
    want = oracle_tree(xh, N)
    fused = lambda bufs: ddp.tree_allreduce_fused(bufs, N)
    for cap in (0, 40):
        prev_kernel = ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_VECTOR)
        prev_cap = ddp.ddp_set_max_ctas(cap)
        try:
            got = run_rank_buffers(fused, xh, f"tree N={N} S={S} cap={cap}")
        finally:
            ddp.ddp_set_max_ctas(prev_cap)
            ddp.ddp_set_fused_kernel(prev_kernel)
        assert_bits_equal(got, want, f"vector tree N={N} S={S} {dtype} cap={cap}")
