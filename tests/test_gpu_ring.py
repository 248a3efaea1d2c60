"""GPU parity of the ring allreduce kernels against the CPU oracle.

Bit-exact comparison (the summation order is fixed, so any difference is a
bug) of ring_allreduce_fused and ring_allreduce_staged, called through the C
ABI, with the oracle's ring simulation on the same seeded inputs:
  * the pages' 3-rank, length-6 example and the order pins;
  * every N in 1..9 with every S in 0..70 (ragged chunks, empty chunks);
  * sizes spanning many tiles with ragged tails, both dtypes, several divisors;
  * buffers that are not 16-byte aligned (element-wise path);
  * the N=4, 1 Mi-element fp32 bucket and the sweep points up to 1 MiB per
    rank (full comparison; the full-size buckets are in test_gpu_full_ring.py).
Tolerance against float64: normwise 1e-5 (fp32) and 2e-2 (bf16).
"""
import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import (assert_bits_equal, assert_canaries, f32_or_bits, from_np, guarded_copy, oracle_allreduce,
                      run_rank_buffers)

pytestmark = pytest.mark.gpu

def _persistent(x, divisor):
    st = ddp.ring_allreduce_persistent(x, divisor)
    torch.cuda.synchronize()
    assert int(st[0]) == 0, f"persistent ring status {int(st[0])}"


KERNELS = {"fused": ddp.ring_allreduce_fused, "staged": ddp.ring_allreduce_staged, "persistent": _persistent}


def run_gpu(kernel: str, x_host: np.ndarray, divisor: int) -> np.ndarray:
    storage, x = guarded_copy(from_np(x_host))
    KERNELS[kernel](x, divisor)
    torch.cuda.synchronize()
    assert_canaries(storage, f"{kernel} {tuple(x.shape)}")
    return f32_or_bits(x)


FUSED_KINDS = {"auto": ddp.DDP_FUSED_AUTO, "vector": ddp.DDP_FUSED_VECTOR, "group": ddp.DDP_FUSED_GROUP,
               "tma": ddp.DDP_FUSED_TMA}


def _with_fused_kernel(kind, fn):
    prev = ddp.ddp_set_fused_kernel(FUSED_KINDS[kind])
    try:
        return fn()
    finally:
        ddp.ddp_set_fused_kernel(prev)


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_worked_example(kernel):
    k = np.arange(6, dtype=np.float32)
    x = np.stack([k + 1, 10 * (k + 1), 100 * (k + 1)]).astype(np.float32)
    got = run_gpu(kernel, x, 3)
    want = np.tile((37 * (k + 1)).astype(np.float32), (3, 1))
    assert_bits_equal(got, want, kernel)
    assert_bits_equal(got, oracle_allreduce(x, 3), kernel)


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_order_pins(kernel):
    for N in (3, 4):
        x = np.zeros((N, N), dtype=np.float32)
        for j in range(N):
            x[(j + 1) % N, j] = 2.0 ** 24
            x[(j + 2) % N, j] = 1.0
            if N == 4:
                x[(j + 3) % N, j] = 1.0
            x[j, j] = -(2.0 ** 24)
        assert np.all(run_gpu(kernel, x, 0) == 0.0)
    f = np.zeros((3, 3), dtype=np.float32)
    for j in range(3):
        f[(j + 1) % 3, j], f[(j + 2) % 3, j], f[j, j] = 256.0, 3.0, -256.0
    got = run_gpu(kernel, oracle.bf16_rne(f), 0)
    assert np.all(oracle.bf16_to_f32(got) == 4.0)


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_exhaustive_small(kernel, dtype):
    for N in range(1, 10):
        for S in range(0, 71):
            x = workloads.rank_vectors(N, S, "randn", dtype=dtype, seed0=N * 1000 + S)
            xh = f32_or_bits(x)
            for div in (0, N):
                assert_bits_equal(run_gpu(kernel, xh, div), oracle_allreduce(xh, div), f"{kernel} N={N} S={S}")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,S,div", [(2, 1_000_003, 2), (3, 3 * 65536 + 5, 3), (5, 777_777, 5), (7, 1 << 20, 7),
                                     (8, (1 << 21) + 13, 8), (16, 1_048_583, 16), (6, 99_991, 0), (4, 4096, 1)])
def test_many_tiles_ragged(kernel, dtype, N, S, div):
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=17)
    xh = f32_or_bits(x)
    assert_bits_equal(run_gpu(kernel, xh, div), oracle_allreduce(xh, div), f"{kernel} {dtype} N={N} S={S}")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_buffers_take_elementwise_path(kernel, dtype):
    # rank rows start 1 element into 16-byte-aligned storage: element aligned
    # but not 16-byte aligned, so the library takes its element-wise kernels
    N, S = 5, 12_345
    x = workloads.rank_vectors(N, S, "randn", dtype=dtype, seed0=3)
    xh = f32_or_bits(x)
    store = torch.zeros((N, S + 8), dtype=x.dtype, device="cuda")
    rows = [store[r, 1:1 + S] for r in range(N)]
    for r in range(N):
        rows[r].copy_(x[r].cuda())
    KERNELS[kernel](rows, N)
    torch.cuda.synchronize()
    got = np.stack([f32_or_bits(r) for r in rows])
    assert_bits_equal(got, oracle_allreduce(xh, N), kernel)


@pytest.mark.parametrize("N,S,dtype", [
    (5, 5 * 262144 - 4, "f32"),      # chunks of 262144, last chunk 4 shorter
    (9, 9 * 131072 - 8, "bf16"),     # chunks of 131072, last chunk 8 shorter
    (64, 64 * 16384 - 60, "f32"),    # 64 ranks, last chunk 60 shorter
    (2, 1 << 22, "bf16"),            # two ranks, equal chunks
    (1, 1 << 21, "f32"),             # one rank: divide only
])
def test_tma_staged_path_ragged_last_chunk(N, S, dtype):
    # 16-byte aligned chunks and bucket, several MiB over all ranks: the TMA
    # kernel streams tiles through shared memory with bulk copies; tiles stop
    # at chunk ends, so chunk ends that are not tile multiples are hit.  The
    # size-based choice runs the same call too.
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=N + 40)
    xh = f32_or_bits(x)
    es = 2 if dtype == "bf16" else 4
    clen = -(-S // N)
    assert (clen * es) % 16 == 0 and (S * es) % 16 == 0 and S * es * N >= 4 << 20
    for div in (N, 0):
        want = oracle_allreduce(xh, div)
        for kind in ("tma", "auto"):
            got = _with_fused_kernel(kind, lambda: run_gpu("fused", xh, div))
            assert_bits_equal(got, want, f"{kind} N={N} S={S} {dtype} div={div}")
    assert ddp.ddp_device_status() == 0


def test_tma_alternating_world_sizes():
    # the TMA kernel needs a different amount of shared memory per world
    # size; calls that alternate between larger and smaller needs on the same
    # kernel must all launch and stay exact
    for N, S in ((8, 1 << 20), (4, 1 << 20), (8, 1 << 20), (2, 1 << 21), (16, 1 << 19), (8, 1 << 20)):
        x = workloads.rank_vectors(N, S, "randn", seed0=N).numpy()
        got = _with_fused_kernel("tma", lambda: run_gpu("fused", x, N))
        assert_bits_equal(got, oracle_allreduce(x, N), f"N={N}")


def test_staged_equals_fused_bitwise_random_shapes():
    rng = np.random.default_rng(0)
    for _ in range(25):
        N = int(rng.integers(1, 20))
        S = int(rng.integers(0, 200_000))
        dtype = "bf16" if rng.integers(0, 2) else "f32"
        x = workloads.rank_vectors(N, S, "uniform", dtype=dtype, seed0=int(rng.integers(0, 1000))).cuda()
        a, b = x.clone(), x.clone()
        ddp.ring_allreduce_fused(a, N)
        ddp.ring_allreduce_staged(b, N)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16) if dtype == "bf16" else a.view(torch.int32),
                           b.view(torch.int16) if dtype == "bf16" else b.view(torch.int32))


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_config_n4_one_mi_fp32_full(kernel):
    # one bucket of 1,048,576 fp32 per rank, N(0,1) from seed r, divide by 4
    N, S = 4, 1 << 20
    x = workloads.rank_vectors(N, S, "randn")
    xh = x.numpy()
    got = run_gpu(kernel, xh, 4)
    want = oracle_allreduce(xh, 4)
    assert_bits_equal(got, want, kernel)
    s64 = xh.astype(np.float64).sum(0) / 4
    assert np.linalg.norm(got[0] - s64) / np.linalg.norm(s64) <= 1e-5


@pytest.mark.parametrize("N", [8, 64])
@pytest.mark.parametrize("kb", [4, 64, 1024])
def test_message_size_sweep(N, kb):
    # uniform(-1,1) fp32, S_b = kb KiB per rank; the 16 MiB and 256 MiB
    # points are compared in full in test_gpu_full_ring.py
    S = kb * 1024 // 4
    x = workloads.rank_vectors(N, S, "uniform").numpy()
    for kernel in ("fused", "staged", "persistent"):
        assert_bits_equal(run_gpu(kernel, x, N), oracle_allreduce(x, N), f"{kernel} N={N} {kb}KiB")


def test_accumulate_matches_oracle():
    for dtype in ("f32", "bf16"):
        for N, S in ((1, 5), (3, 1001), (8, 1 << 20)):
            a = workloads.rank_vectors(N, S, "randn", dtype=dtype, seed0=1)
            g = workloads.rank_vectors(N, S, "randn", dtype=dtype, seed0=100)
            ah, gh = f32_or_bits(a), f32_or_bits(g)
            ad, gd = a.cuda(), g.cuda()
            ddp.ddp_grad_accumulate(ad, gd)
            torch.cuda.synchronize()
            want = ah.copy()
            code = oracle.BF16 if dtype == "bf16" else oracle.F32
            for r in range(N):
                oracle.accumulate(want[r], gh[r], code)
            assert_bits_equal(f32_or_bits(ad), want, f"accumulate {dtype} N={N} S={S}")


def test_from_host_matches_oracle():
    N, S = 8, 1_000_001
    x = workloads.rank_vectors(N, S, "randn", seed0=5)
    want = oracle_allreduce(x.numpy(), 8)
    host_in = x.pin_memory()
    host_out = torch.empty_like(host_in).pin_memory()
    dev = torch.empty((N, S), dtype=torch.float32, device="cuda")
    ddp.ring_allreduce_fused_from_host(host_in, host_out, dev, 8)
    torch.cuda.synchronize()
    assert_bits_equal(host_out.numpy(), want, "from_host")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("alias", [False, True])
def test_from_host_pipelined_in_pieces_matches_oracle(dtype, alias):
    # more than two 32 MiB pieces per rank, ragged last piece and chunk
    # boundaries inside pieces: the pieces are reduced on internal streams
    # while others are copied in and out; host_out may be host_in
    es = 2 if dtype == "bf16" else 4
    N, S = 3, (5 * (32 << 20)) // es + 12_345
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=61)
    xh = f32_or_bits(x)
    want = oracle_allreduce(xh, N)
    host_in = x.pin_memory()
    host_out = host_in if alias else torch.empty_like(host_in).pin_memory()
    dev = torch.empty((N, S), dtype=x.dtype, device="cuda")
    stream = torch.cuda.Stream()
    ddp.ring_allreduce_fused_from_host(host_in, host_out, dev, N, stream=stream)
    stream.synchronize()
    assert_bits_equal(f32_or_bits(host_out), want, f"from_host pieces {dtype} alias={alias}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,S", [(3, 6), (8, 1_000_001), (4, 1 << 20), (16, 77_777)])
def test_host_direct_matches_oracle(dtype, N, S):
    # the kernel reads pinned host memory and writes the result back to it
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=N + 7)
    xh = f32_or_bits(x)
    want = oracle_allreduce(xh, N)
    src = x.pin_memory()
    out = torch.zeros_like(src).pin_memory()
    ddp.ring_allreduce_fused_host_direct(src, out, N)           # out of place
    torch.cuda.synchronize()
    assert_bits_equal(f32_or_bits(out), want, "host direct out of place")
    assert_bits_equal(f32_or_bits(src), xh, "host direct input untouched")
    ddp.ring_allreduce_fused_host_direct(src, src, N)           # in place
    torch.cuda.synchronize()
    assert_bits_equal(f32_or_bits(src), want, "host direct in place")


def test_host_direct_unaligned_and_pageable():
    N, S = 5, 10_001
    x = workloads.rank_vectors(N, S, "randn", seed0=2)
    want = oracle_allreduce(x.numpy(), N)
    store = torch.zeros((N, S + 4)).pin_memory()
    rows = [store[r, 1:1 + S] for r in range(N)]                # 4-byte but not 16-byte aligned
    for r in range(N):
        rows[r].copy_(x[r])
    ddp.ring_allreduce_fused_host_direct(rows, rows, N)
    torch.cuda.synchronize()
    assert_bits_equal(np.stack([r.numpy() for r in rows]), want, "unaligned pinned")
    pageable = x.clone()
    try:
        ddp.ring_allreduce_fused_host_direct(pageable, pageable, N)
    except ddp.DDPError as e:
        assert e.status == -1                                    # this GPU cannot read pageable memory
    else:
        torch.cuda.synchronize()
        assert_bits_equal(pageable.numpy(), want, "pageable")


def test_persistent_barrier_timeout_is_reported_and_context_survives():
    # a planted missing arrival at the barrier ending step 1: every block
    # waits 200 ms, reports DDP_ERR_TIMEOUT and returns
    import time
    N, S = 4, 1 << 16
    x = workloads.rank_vectors(N, S, "randn", seed0=9).cuda()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = ddp.ring_allreduce_persistent(x, N, fail_at_step=1, wait_limit_ms=200)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st[0]) == -4
    assert 0.15 < dt < 5.0
    # the context is still usable and exact afterwards
    y = workloads.rank_vectors(N, S, "randn", seed0=10).numpy()
    for kernel in ("fused", "persistent"):
        assert_bits_equal(run_gpu(kernel, y, N), oracle_allreduce(y, N), f"after timeout: {kernel}")


def test_persistent_status_word_is_cleared_on_each_call():
    N, S = 3, 1000
    x = workloads.rank_vectors(N, S, "randn", seed0=1).cuda()
    st = torch.full((2,), -4, dtype=torch.int32, device="cuda")
    ddp.ring_allreduce_persistent(x, N, status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0


@pytest.mark.parametrize("cap", [1, 7, 40])
def test_cta_cap_does_not_change_results(cap):
    # every kernel family under a CTA cap: each fused kernel (TMA, group and
    # vector on aligned buckets, element-wise on ragged ones), staged,
    # persistent -- all must stay exact
    cases = [(8, 1 << 20, "f32"), (5, 77_777, "bf16"), (3, 1000, "f32")]
    prev = ddp.ddp_set_max_ctas(cap)
    try:
        for N, S, dtype in cases:
            x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=cap + N)
            xh = f32_or_bits(x)
            want = oracle_allreduce(xh, N)
            for kind in ("tma", "group", "vector"):
                got = _with_fused_kernel(kind, lambda: run_gpu("fused", xh, N))
                assert_bits_equal(got, want, f"cap={cap} fused/{kind} N={N} S={S}")
            for kernel in ("staged", "persistent"):
                assert_bits_equal(run_gpu(kernel, xh, N), want, f"cap={cap} {kernel} N={N} S={S}")
    finally:
        ddp.ddp_set_max_ctas(prev)


# Buckets of at least 128 MiB over all ranks run the vector kernel with one
# block per tile of vectors (two vectors per thread over 2 or 3 ranks); a CTA
# cap below the tile count makes the same launch loop over its tiles.  The
# sizes leave chunk boundaries off the 16-byte grid and a ragged last vector;
# each rank has its own 16-byte-aligned buffer, so the vector kernel runs.
STREAMED = [(2, 16_777_219), (3, 11_184_813), (5, 6_710_891), (8, 4_194_307), (12, 2_796_205)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,S", STREAMED)
def test_vector_kernel_one_block_per_tile(dtype, N, S):
    S = S * 2 if dtype == "bf16" else S
    assert N * S * (2 if dtype == "bf16" else 4) >= 128 << 20
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=11 * N)
    xh = f32_or_bits(x)
    want = oracle_allreduce(xh, N)
    fused = lambda bufs: ddp.ring_allreduce_fused(bufs, N)
    got = _with_fused_kernel("vector", lambda: run_rank_buffers(fused, xh, f"ring N={N} S={S}"))
    assert_bits_equal(got, want, f"vector one block per tile N={N} S={S} {dtype}")
    prev = ddp.ddp_set_max_ctas(40)
    try:
        got = _with_fused_kernel("vector", lambda: run_rank_buffers(fused, xh, f"ring N={N} S={S} cap 40"))
    finally:
        ddp.ddp_set_max_ctas(prev)
    assert_bits_equal(got, want, f"vector, 40 blocks looping over the tiles, N={N} S={S} {dtype}")


def test_empty_bucket_is_noop():
    x = torch.zeros((4, 0), device="cuda")
    ddp.ring_allreduce_fused(x, 4)
    ddp.ring_allreduce_staged(x, 4)
    st = ddp.ring_allreduce_persistent(x, 4)
    torch.cuda.synchronize()
    assert int(st[0]) == 0


def test_single_rank_divides_only():
    x = workloads.rank_vectors(1, 1003, "randn").numpy()
    for kernel in ("fused", "staged"):
        assert_bits_equal(run_gpu(kernel, x, 3), oracle_allreduce(x, 3), kernel)
        assert_bits_equal(run_gpu(kernel, x, 0), x, kernel)


@pytest.mark.parametrize("kind", ["vector", "group", "tma", "auto"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_fused_kernel_matches_oracle(kind, dtype):
    # each fused kernel forced on world sizes that exercise every lane split
    # of the group kernel (P = 2 .. 32 lanes per vector, 1, 2 or 4 vectors
    # per lane) and the fallbacks (N = 1, N > 128); sizes with straddling
    # vectors (chunk not a multiple of the vector), ragged tails, chunk
    # multiples of 16 bytes (TMA-eligible) and several tiles
    es = 2 if dtype == "bf16" else 4
    per16 = 16 // es
    cases = []
    for N in (1, 2, 3, 4, 5, 8, 9, 16, 17, 31, 32, 33, 63, 64, 65, 100, 128, 130):
        cases += [(N, 7 * N + 3), (N, N * per16 * 37), (N, N * per16 * 1024 + 5 * per16)]
    cases += [(8, 8 * per16 * 5000), (64, 64 * per16 * 300 + 11), (3, 1_000_003)]
    for i, (N, S) in enumerate(cases):
        x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=100 + i)
        xh = f32_or_bits(x)
        for div in ((N, 0, 3) if i % 3 == 0 else (N,)):
            got = _with_fused_kernel(kind, lambda: run_gpu("fused", xh, div))
            assert_bits_equal(got, oracle_allreduce(xh, div), f"{kind} {dtype} N={N} S={S} div={div}")


@pytest.mark.parametrize("kind", ["vector", "group", "tma"])
def test_forced_fused_kernel_on_unaligned_buffers_falls_back(kind):
    # a forced kernel that cannot run the call (rows not 16-byte aligned)
    # gives way to the element-wise kernel, with the same result
    N, S = 6, 4099
    x = workloads.rank_vectors(N, S, "randn", seed0=5)
    xh = f32_or_bits(x)
    store = torch.zeros((N, S + 8), dtype=x.dtype, device="cuda")
    rows = [store[r, 1:1 + S] for r in range(N)]
    for r in range(N):
        rows[r].copy_(x[r].cuda())
    _with_fused_kernel(kind, lambda: ddp.ring_allreduce_fused(rows, N))
    torch.cuda.synchronize()
    assert_bits_equal(np.stack([f32_or_bits(r) for r in rows]), oracle_allreduce(xh, N), kind)


@pytest.mark.parametrize("kind", ["vector", "group", "tma"])
def test_forced_fused_kernel_in_bucketed_sync(kind):
    # the bucketed DDP step (pack + fused ring + unpack) is the same whichever
    # kernel reduces the buckets
    from test_gpu_buckets import _device_views, _host_grads, _small_decoder
    numels = _small_decoder()
    world, first, cap = 8, 4096, 40000
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, first, cap)
    flat, grads_h = _host_grads(numels, world, "f32", seed0=21)
    g = flat.cuda()
    views = _device_views(g, numels)
    bk = [[torch.empty(int(n), dtype=torch.float32, device="cuda") for n in plan[2]] for _ in range(world)]
    _with_fused_kernel(kind, lambda: ddp.ddp_sync_buckets(views, plan, bk, algo=ddp.DDP_ALGO_FUSED))
    torch.cuda.synchronize()
    oracle.ddp_sync(grads_h, oracle.F32, first, cap)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"bucketed sync with {kind}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_maximum_world_size(dtype):
    # DDP_MAX_WORLD = 512 ranks on a ragged bucket (chunks of 5 elements, the
    # last ones short or empty): every ring kernel, the staged tree and the
    # view sync of a 3-member bucket
    N, S = 512, 2053
    xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=9))
    want = oracle_allreduce(xh, N)
    for kernel in ("fused", "staged", "persistent"):
        assert_bits_equal(run_gpu(kernel, xh, N), want, f"{kernel} N={N}")
    x = from_np(xh)
    ddp.tree_allreduce_staged(x, N)
    torch.cuda.synchronize()
    t = np.ascontiguousarray(xh).copy()
    oracle.tree_allreduce_2d(t, oracle.BF16 if dtype == "bf16" else oracle.F32, N)
    assert_bits_equal(f32_or_bits(x), t, "tree staged N=512")
    # view: members of 1000, 53 and 1000 elements at bucket offsets 0, 1000, 1053
    x = from_np(xh)
    numels, offsets = [1000, 53, 1000], [0, 1000, 1053]
    views = [[x[r, o:o + n] for o, n in zip(offsets, numels)] for r in range(N)]
    ddp.ddp_bucket_allreduce_view(views, offsets, S, N)
    torch.cuda.synchronize()
    assert_bits_equal(f32_or_bits(x), want, "view N=512")

