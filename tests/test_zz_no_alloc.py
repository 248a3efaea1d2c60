"""The allocation-free host-buffer allreduce.

ring_allreduce_fused_from_host_noalloc is for callers that hold gradients in
host memory and cannot allocate device memory themselves (no device
allocator of their own, or one that belongs to another framework).  It
keeps the ranks' device copies in a fixed array that the library reserves
on every GPU.  Call after call, whatever the previous call left in that
shared array, it must give the CPU oracle's ring result bit for bit (the
bar of every other parity test here), and so exactly what
ring_allreduce_fused_from_host gives with caller-allocated device buffers.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import workloads
from gpu_util import assert_bits_equal, f32_or_bits, oracle_allreduce


def _pinned(x):
    return x.contiguous().pin_memory()


@pytest.mark.gpu
def test_noalloc_matches_caller_allocated_variant_on_consecutive_calls():
    # consecutive calls with different shapes and dtypes: the second and
    # third calls find the previous call's data in the shared array
    cases = [(8, 1_000_003, "f32", 11), (4, 1 << 20, "bf16", 12), (8, 1_000_003, "f32", 13), (3, 5, "f32", 14)]
    for N, S, dtype, seed in cases:
        x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=seed)
        host_in = _pinned(x)
        want = torch.empty_like(host_in).pin_memory()
        got = torch.empty_like(host_in).pin_memory()
        dev = torch.empty((N, S), dtype=x.dtype, device="cuda")
        ddp.ring_allreduce_fused_from_host(host_in, want, dev, N)
        ddp.ring_allreduce_fused_from_host_noalloc(host_in, got, N)
        torch.cuda.synchronize()
        iv = torch.int16 if dtype == "bf16" else torch.int32
        assert_bits_equal(f32_or_bits(got), oracle_allreduce(f32_or_bits(x), N), f"oracle N={N} S={S} {dtype}")
        assert torch.equal(got.view(iv), want.view(iv)), f"N={N} S={S} {dtype}"
        # the input buffers are left untouched when host_out differs
        assert torch.equal(host_in.view(iv), x.view(iv))


@pytest.mark.gpu
def test_noalloc_in_place_on_host():
    N, S = 5, 777_777
    x = workloads.rank_vectors(N, S, "randn", seed0=3)
    a = _pinned(x)
    b = torch.empty_like(a).pin_memory()
    dev = torch.empty((N, S), device="cuda")
    want = oracle_allreduce(x.numpy(), N)
    ddp.ring_allreduce_fused_from_host(a, b, dev, N)
    ddp.ring_allreduce_fused_from_host_noalloc(a, a, N)       # host_out == host_in
    torch.cuda.synchronize()
    assert_bits_equal(a.numpy(), want, "noalloc in place")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_noalloc_rejects_requests_beyond_the_array_before_any_cuda_call():
    L = ddp.lib()
    H = 0x7f0000000000                       # never dereferenced: every call below is refused
    tab = (ctypes.c_void_p * 8)(*[H + r * (1 << 27) for r in range(8)])    # 128 MiB apart: disjoint
    limit = ddp.STATIC_SCRATCH_BYTES
    # 8 ranks x (limit / 8 + 4 bytes) of fp32 does not fit
    assert L.ring_allreduce_fused_from_host_noalloc(8, tab, tab, limit // 32 + 1, 0, 8, None) == -5
    # one rank larger than the whole array
    assert L.ring_allreduce_fused_from_host_noalloc(1, tab, tab, limit // 4 + 1, 0, 1, None) == -5
    # rounding each rank up to 256 bytes is counted: 3 ranks of 11,184,810
    # bf16 fit unrounded (67,108,860 bytes) but not rounded (67,109,376)
    assert 3 * 11_184_810 * 2 <= limit < 3 * ((11_184_810 * 2 + 255) // 256 * 256)
    assert L.ring_allreduce_fused_from_host_noalloc(3, tab, tab, 11_184_810, 1, 3, None) == -5
    assert L.ring_allreduce_fused_from_host_noalloc(8, None, tab, 16, 0, 8, None) == -1
    assert L.ring_allreduce_fused_from_host_noalloc(0, tab, tab, 16, 0, 8, None) == -1
    assert L.ring_allreduce_fused_from_host_noalloc(8, tab, tab, 16, 7, 8, None) == -1
    assert L.ring_allreduce_fused_from_host_noalloc(8, tab, tab, 0, 0, 8, None) == 0    # empty: no CUDA work
    with pytest.raises(ddp.DDPError):
        ddp.ring_allreduce_fused_from_host_noalloc(torch.zeros(2, limit // 8 + 64), torch.zeros(2, limit // 8 + 64), 2,
                                                   stream=0)


@pytest.mark.skipif(torch.cuda.is_available(), reason="refusals with made-up pointers run only where no GPU is reachable")
def test_noalloc_rejects_sizes_whose_byte_count_would_overflow():
    # numel * element size must never be formed for a numel beyond
    # DDP_MAX_NUMEL: 2^62 + 16 fp32 elements are 2^64 + 64 bytes, which wraps
    # to 64 bytes in 64-bit arithmetic and would pass a capacity check made on
    # the wrapped value.  Every call here must be refused before any CUDA
    # call; this test runs only without a GPU, so a regression cannot reach
    # a copy or a launch.
    L = ddp.lib()
    H = 0x7f0000000000
    tab = (ctypes.c_void_p * 8)(*[H + r * (1 << 27) for r in range(8)])
    for numel in ((1 << 62) + 16, (1 << 62) + 8, (1 << 63) - 1, ddp.MAX_NUMEL + 1):
        for dtype in (0, 1):
            for world in (1, 2, 8):
                assert L.ring_allreduce_fused_from_host_noalloc(world, tab, tab, numel, dtype, world, None) == -5
    # within DDP_MAX_NUMEL but beyond the array: refused by the capacity check
    assert L.ring_allreduce_fused_from_host_noalloc(1, tab, tab, ddp.MAX_NUMEL, 0, 1, None) == -5
