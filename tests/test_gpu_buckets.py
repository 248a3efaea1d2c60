"""GPU parity of the bucket path: plan -> pack -> ring allreduce / N -> unpack.

Against the oracle's own composition of the same steps (``oracle.ddp_sync``,
``oracle.no_sync_then_sync``), bit-exact, through the C ABI:
  * pack/unpack of random member lists with odd sizes and offsets (so slots
    are often not 16-byte aligned), both dtypes;
  * ddp_sync_buckets with each algorithm (fused, staged, fused view) on a
    small decoder with many buckets, and the view kernel against
    pack + fused + unpack;
  * the ResNet-50 parameter list in bf16, N = 16, caps 5/10/25/50 MiB (full
    comparison);
  * (the 355M-parameter decoder at full size is in test_gpu_full_decoder.py);
  * buckets larger than L2, which the unfused path runs in L2-sized pieces:
    members straddling piece and chunk boundaries, and sizes on both sides
    of the switch between whole buckets and pieces.
"""
import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import assert_bits_equal, assert_canaries, f32_or_bits, guarded_copy, oracle_allreduce

pytestmark = pytest.mark.gpu
MiB = 1 << 20


def _host_grads(numels, world, dtype, seed0, kind="randn", std=1e-2):
    """grads[r][p] host arrays (float32 or uint16 bf16 bits), rank r from seed seed0+r."""
    total = sum(numels)
    flat = workloads.rank_vectors(world, total, kind, std=std, dtype=dtype, seed0=seed0)
    flat_h = f32_or_bits(flat)
    out, o = [], 0
    offs = np.cumsum([0] + list(numels))
    return flat, [[flat_h[r, offs[p]:offs[p + 1]].copy() for p in range(len(numels))] for r in range(world)]


# Segment tables of the view path are folded by the TMA-staged view kernel or
# by the register view kernel (ddp_set_fused_kernel: TMA, or vector); "auto"
# picks by size, "vector_cap" forces the register kernel under a CTA cap so
# that its blocks loop over the tiles.
VIEW_KERNELS = ["auto", "tma", "vector", "vector_cap"]


class _view_kernel:
    def __init__(self, kind):
        self.kind = kind

    def __enter__(self):
        k = {"auto": ddp.DDP_FUSED_AUTO, "tma": ddp.DDP_FUSED_TMA}.get(self.kind, ddp.DDP_FUSED_VECTOR)
        self.prev = ddp.ddp_set_fused_kernel(k)
        self.prev_cap = ddp.ddp_set_max_ctas(40) if self.kind == "vector_cap" else None
        return self

    def __exit__(self, *exc):
        ddp.ddp_set_fused_kernel(self.prev)
        if self.prev_cap is not None:
            ddp.ddp_set_max_ctas(self.prev_cap)
        return False


def _device_views(flat_dev, numels):
    offs = np.cumsum([0] + list(numels))
    return [[flat_dev[r, int(offs[p]):int(offs[p + 1])] for p in range(len(numels))]
            for r in range(flat_dev.shape[0])]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pack_unpack_random_members(dtype):
    rng = np.random.default_rng(1)
    for trial in range(20):
        world = int(rng.integers(1, 9))
        n = int(rng.integers(1, 30))
        numels = [int(v) for v in rng.integers(0, 5000, size=n)]
        code = oracle.BF16 if dtype == "bf16" else oracle.F32
        order = list(rng.permutation(n))
        offsets, pos = [0] * n, int(rng.integers(0, 7))
        for i in order:
            offsets[i] = pos
            pos += numels[i] + int(rng.integers(0, 3))
        bucket_numel = pos + int(rng.integers(0, 5))
        flat, grads_h = _host_grads(numels, world, dtype, seed0=trial * 10)
        gdev = _device_views(flat.cuda(), numels)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        buckets = torch.zeros((world, bucket_numel), dtype=tdt, device="cuda")
        ddp.ddp_bucket_pack(gdev, offsets, buckets)
        torch.cuda.synchronize()
        want = np.zeros((world, bucket_numel), dtype=np.uint16 if dtype == "bf16" else np.float32)
        for r in range(world):
            oracle.bucket_pack(grads_h[r], offsets, want[r], code)
        assert_bits_equal(f32_or_bits(buckets), want, f"pack trial {trial}")
        # unpack a different bucket content back into zeroed gradients
        src = workloads.rank_vectors(world, bucket_numel, "uniform", dtype=dtype, seed0=99 + trial)
        src_h = f32_or_bits(src)
        out = [[torch.zeros_like(g) for g in gdev[r]] for r in range(world)]
        ddp.ddp_bucket_unpack(out, offsets, src.cuda())
        torch.cuda.synchronize()
        for r in range(world):
            exp = [np.zeros_like(g) for g in grads_h[r]]
            oracle.bucket_unpack(exp, offsets, src_h[r], code)
            for i in range(n):
                assert_bits_equal(f32_or_bits(out[r][i]), exp[i], f"unpack trial {trial} r{r} m{i}")


def _small_decoder():
    return workloads.param_numels(workloads.decoder_param_shapes(n_layer=3, d_model=64, d_ff=256, vocab=1000,
                                                                 n_pos=64))


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_STAGED, ddp.DDP_ALGO_VIEW])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sync_buckets_small_decoder(algo, dtype):
    numels = _small_decoder()
    world = 8
    es = 2 if dtype == "bf16" else 4
    first, cap = 4096, 40000
    plan = ddp.ddp_plan_buckets(numels, ddp.BF16 if dtype == "bf16" else ddp.F32, first, cap)
    assert len(plan[2]) > 5
    flat, grads_h = _host_grads(numels, world, dtype, seed0=0)
    g_storage, gdev_flat = guarded_copy(flat)
    gdev = _device_views(gdev_flat, numels)
    bk = None
    if algo != ddp.DDP_ALGO_VIEW:
        bk = [[torch.empty(int(n), dtype=flat.dtype, device="cuda") for n in plan[2]] for _ in range(world)]
    ddp.ddp_sync_buckets(gdev, plan, bk, algo=algo)
    torch.cuda.synchronize()
    assert_canaries(g_storage, f"small decoder algo={algo}")
    oracle.ddp_sync(grads_h, oracle.BF16 if dtype == "bf16" else oracle.F32, first, cap)
    got = f32_or_bits(gdev_flat)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(got, want, f"sync algo={algo} {dtype}")
    assert es in (2, 4)


def test_view_equals_pack_fused_unpack_bitwise():
    rng = np.random.default_rng(3)
    for trial in range(12):
        world = int(rng.integers(1, 17))
        n = int(rng.integers(1, 12))
        numels = [int(v) for v in rng.integers(1, 20000, size=n)]
        dtype = "bf16" if trial % 2 else "f32"
        b_of, off, bn = ddp.ddp_plan_buckets(numels, ddp.BF16 if dtype == "bf16" else ddp.F32, 10 ** 9, 10 ** 9)
        assert len(bn) == 1
        flat = workloads.rank_vectors(world, sum(numels), "randn", dtype=dtype, seed0=trial).cuda()
        a, b = flat.clone(), flat.clone()
        ga, gb = _device_views(a, numels), _device_views(b, numels)
        offsets = [int(o) for o in off]
        ddp.ddp_bucket_allreduce_view(ga, offsets, int(bn[0]), world)
        bucket = torch.empty((world, int(bn[0])), dtype=flat.dtype, device="cuda")
        ddp.ddp_bucket_pack(gb, offsets, bucket)
        ddp.ring_allreduce_fused(bucket, world)
        ddp.ddp_bucket_unpack(gb, offsets, bucket)
        torch.cuda.synchronize()
        iv = torch.int16 if dtype == "bf16" else torch.int32
        assert torch.equal(a.view(iv), b.view(iv)), f"trial {trial}"


@pytest.mark.parametrize("kernel", ["auto", "tma"])
@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_VIEW])
@pytest.mark.parametrize("cap_mib,count", [(5, 9), (10, 6), (25, 3), (50, 2)])
def test_resnet50_bf16_n16_cap_sweep_full(cap_mib, count, algo, kernel):
    # pack + fused ring + unpack, and the fused view (one launch of the
    # register view kernel, one block per tile, by size -- or of the TMA view
    # kernel, forced -- whose threads also fold the elements around the fc
    # bucket's unaligned chunk boundaries)
    numels = workloads.param_numels(workloads.resnet50_param_shapes())
    world = 16
    plan = ddp.ddp_plan_buckets(numels, ddp.BF16, MiB, cap_mib * MiB)
    assert len(plan[2]) == count
    flat, grads_h = _host_grads(numels, world, "bf16", seed0=0)
    g_storage, gdev_flat = guarded_copy(flat)
    gdev = _device_views(gdev_flat, numels)
    bk = None
    if algo == ddp.DDP_ALGO_FUSED:
        bk = [[torch.empty(int(n), dtype=torch.bfloat16, device="cuda") for n in plan[2]] for _ in range(world)]
    with _view_kernel(kernel):
        ddp.ddp_sync_buckets(gdev, plan, bk, algo=algo)
    torch.cuda.synchronize()
    assert_canaries(g_storage, f"resnet50 cap {cap_mib} algo {algo} kernel {kernel}")
    ref64 = np.zeros(sum(numels))
    for r in range(world):
        ref64 += oracle.bf16_to_f32(np.concatenate(grads_h[r])).astype(np.float64)
    ref64 /= world
    oracle.ddp_sync(grads_h, oracle.BF16, MiB, cap_mib * MiB)
    got = f32_or_bits(gdev_flat)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(got, want, f"resnet50 cap {cap_mib} algo {algo}")
    y = oracle.bf16_to_f32(got[0]).astype(np.float64)
    assert np.linalg.norm(y - ref64) / np.linalg.norm(ref64) <= 2e-2


def test_no_sync_small_decoder_full():
    numels = _small_decoder()
    world, M = 4, 4
    micro_h, micro_d = [], []
    for m in range(M):
        rows = [workloads.randn_f32(sum(numels), workloads.microbatch_seed(r, world, m), 1e-2) for r in range(world)]
        flat = torch.stack(rows)
        offs = np.cumsum([0] + numels)
        micro_h.append([[flat[r, offs[p]:offs[p + 1]].numpy().copy() for p in range(len(numels))]
                        for r in range(world)])
        micro_d.append(flat.cuda())
    acc = micro_d[0].clone()
    for m in range(1, M):
        ddp.ddp_grad_accumulate(acc, micro_d[m])
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, 4096, 40000)
    gdev = _device_views(acc, numels)
    ddp.ddp_sync_buckets(gdev, plan, None, algo=ddp.DDP_ALGO_VIEW)
    torch.cuda.synchronize()
    want = oracle.no_sync_then_sync(micro_h, oracle.F32, 4096, 40000)
    assert_bits_equal(f32_or_bits(acc), np.stack([np.concatenate(want[r]) for r in range(world)]), "no_sync")


@pytest.mark.parametrize("algo", ["hook", "hook_view", "fp16_hook_view"])
@pytest.mark.parametrize("via", ["sync_buckets", "reducer"])
def test_bf16_hook_matches_oracle(via, algo):
    numels = _small_decoder()
    world, first, cap = 8, 4096, 40000
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, first, cap)
    flat, grads_h = _host_grads(numels, world, "f32", seed0=4)
    x64 = flat.numpy().astype(np.float64)
    g = flat.cuda()
    views = _device_views(g, numels)
    code = {"hook": ddp.DDP_ALGO_BF16_HOOK, "hook_view": ddp.DDP_ALGO_BF16_HOOK_VIEW,
            "fp16_hook_view": ddp.DDP_ALGO_FP16_HOOK_VIEW}[algo]
    bk = None
    if algo == "hook":
        bk = [[torch.empty(int(n), dtype=torch.bfloat16, device="cuda") for n in plan[2]] for _ in range(world)]
    if via == "sync_buckets":
        ddp.ddp_sync_buckets(views, plan, bk, algo=code)
    else:
        red = ddp.Reducer(views, plan, bk, algo=code, comm_stream=torch.cuda.Stream())
        for p in range(len(numels) - 1, -1, -1):
            red.mark_ready(p, torch.cuda.current_stream())
        red.finalize(torch.cuda.current_stream())
    torch.cuda.synchronize()
    if algo == "fp16_hook_view":
        oracle.ddp_sync_fp16_hook(grads_h, first, cap)
    else:
        oracle.ddp_sync_bf16_hook(grads_h, first, cap)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    got = f32_or_bits(g)
    assert_bits_equal(got, want, f"{algo} via {via}")
    ref = x64.sum(0) / world
    assert np.linalg.norm(got[0] - ref) / np.linalg.norm(ref) <= 2e-2


def test_bf16_pack_unpack_round_trip_matches_oracle_rounding():
    rng = np.random.default_rng(8)
    world, numels = 3, [1001, 16, 5, 4096]
    offsets = [0, 1001, 1017, 1022]             # odd offsets: element-wise conversion paths too
    bucket_numel = 1022 + 4096
    grads = [[torch.from_numpy(rng.standard_normal(n).astype(np.float32)).cuda() for n in numels] for _ in range(world)]
    buckets = torch.zeros((world, bucket_numel), dtype=torch.bfloat16, device="cuda")
    ddp.ddp_bucket_pack_bf16(grads, offsets, buckets)
    out = [[torch.zeros_like(t) for t in grads[r]] for r in range(world)]
    ddp.ddp_bucket_unpack_bf16(out, offsets, buckets)
    torch.cuda.synchronize()
    for r in range(world):
        for i in range(len(numels)):
            src = grads[r][i].cpu().numpy()
            want_bits = oracle.bf16_rne(src)
            got_bits = f32_or_bits(buckets[r, offsets[i]:offsets[i] + numels[i]])
            assert_bits_equal(got_bits, want_bits, f"pack r{r} m{i}")
            assert_bits_equal(f32_or_bits(out[r][i]), oracle.bf16_to_f32(want_bits), f"unpack r{r} m{i}")


@pytest.mark.parametrize("kernel", VIEW_KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_view_tma_path_matches_oracle(dtype, kernel):
    # one bucket of ~1.2M elements over 8 ranks (> 4 MiB): member sizes and the
    # chunk length are multiples of 16 elements, so the view path streams
    # chunk-aligned segments through shared memory; one member spans several
    # chunks, others end inside a chunk
    world = 8
    numels = [16 * 7, 16 * 40000, 16 * 3, 16 * 25000, 16 * 1000, 16 * 9006]
    total = sum(numels)
    assert (-(-total // world)) % 16 == 0
    code = ddp.BF16 if dtype == "bf16" else ddp.F32
    es = 2 if dtype == "bf16" else 4
    assert total * es * world >= 4 << 20
    plan = ddp.ddp_plan_buckets(numels, code, 1 << 40, 1 << 40)
    assert len(plan[2]) == 1
    flat, grads_h = _host_grads(numels, world, dtype, seed0=6)
    g = flat.cuda()
    with _view_kernel(kernel):
        ddp.ddp_sync_buckets(_device_views(g, numels), plan, None, algo=ddp.DDP_ALGO_VIEW)
    torch.cuda.synchronize()
    oracle.ddp_sync(grads_h, code, 1 << 40, 1 << 40)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"view {kernel} {dtype}")
    assert ddp.ddp_device_status() == 0



@pytest.mark.parametrize("prec", ["bf16", "fp16"])
@pytest.mark.parametrize("divisor", [None, 0, 3])
def test_bf16_hook_view_tma_path_matches_oracle(divisor, prec):
    # the fused hook on one TMA-sized bucket (> 4 MiB of float32 over 8 ranks,
    # chunk-aligned segments), plus the world-size, no-divide and
    # non-power-of-two divisors; the second call on a ragged single member
    # takes the register path
    view_fn = ddp.ddp_bucket_allreduce_view_fp16 if prec == "fp16" else ddp.ddp_bucket_allreduce_view_bf16
    hook_fn = oracle.ddp_sync_fp16_hook if prec == "fp16" else oracle.ddp_sync_bf16_hook
    world = 8
    numels = [16 * 7, 16 * 40000, 16 * 3, 16 * 25000, 16 * 1000, 16 * 9006]
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, 1 << 40, 1 << 40)
    assert len(plan[2]) == 1
    flat, grads_h = _host_grads(numels, world, "f32", seed0=9)
    g = flat.cuda()
    div = world if divisor is None else divisor
    offsets = [int(o) for o in plan[1]]
    view_fn(_device_views(g, numels), offsets, int(plan[2][0]), div)
    torch.cuda.synchronize()
    hook_fn(grads_h, 1 << 40, 1 << 40, divisor=div)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"hook view tma div={div}")
    assert ddp.ddp_device_status() == 0

    numels = [1001]
    flat, grads_h = _host_grads(numels, 3, "f32", seed0=10)
    g = flat.cuda()
    view_fn(_device_views(g, numels), [0], 1001, div)
    torch.cuda.synchronize()
    hook_fn(grads_h, 1 << 40, 1 << 40, divisor=div)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(3)])
    assert_bits_equal(f32_or_bits(g), want, f"hook view ragged div={div}")


def test_bf16_hook_view_world_one_rounds():
    # one rank: no hop, but the hook still rounds every value to bf16
    numels = [4096 + 5]
    flat, grads_h = _host_grads(numels, 1, "f32", seed0=11)
    g = flat.cuda()
    ddp.ddp_bucket_allreduce_view_bf16(_device_views(g, numels), [0], numels[0], 1)
    torch.cuda.synchronize()
    oracle.ddp_sync_bf16_hook(grads_h, 1 << 40, 1 << 40, divisor=1)
    assert_bits_equal(f32_or_bits(g), np.stack([grads_h[0][0]]), "hook view world 1")


@pytest.mark.parametrize("layout", ["decoder", "aligned"])
@pytest.mark.parametrize("algo", ["fused", "view", "hook", "hook_view"])
def test_many_ranks_split_into_several_launches(algo, layout):
    # 128 ranks x ~40 members: the pack / unpack / convert item tables and
    # the view pointer tables overflow one launch's parameter space, so each
    # bucket is done in several launches; the result must not change.  The
    # small decoder's chunks are not 16-byte aligned (register view kernel);
    # the "aligned" list's are (TMA view kernel).
    if layout == "decoder":
        numels = _small_decoder()
    else:
        numels = [512 * (i % 7 + 1) for i in range(40)]
    world, first, cap = 128, 4096, 1 << 30
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, first, cap)
    flat, grads_h = _host_grads(numels, world, "f32", seed0=31)
    g = flat.cuda()
    views = _device_views(g, numels)
    code = {"fused": ddp.DDP_ALGO_FUSED, "view": ddp.DDP_ALGO_VIEW, "hook": ddp.DDP_ALGO_BF16_HOOK,
            "hook_view": ddp.DDP_ALGO_BF16_HOOK_VIEW}[algo]
    bk = None
    if algo in ("fused", "hook"):
        bdt = torch.float32 if algo == "fused" else torch.bfloat16
        bk = [[torch.empty(int(n), dtype=bdt, device="cuda") for n in plan[2]] for _ in range(world)]
    ddp.ddp_sync_buckets(views, plan, bk, algo=code)
    torch.cuda.synchronize()
    if algo in ("hook", "hook_view"):
        oracle.ddp_sync_bf16_hook(grads_h, first, cap)
    else:
        oracle.ddp_sync(grads_h, oracle.F32, first, cap)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"{algo} {layout} at N={world}")


def _oracle_view(grads_h, offsets, bucket_numel, code, divisor):
    """Oracle pack -> ring -> unpack of one bucket (in place on grads_h)."""
    world = len(grads_h)
    dt = np.uint16 if code == oracle.BF16 else np.float32
    bufs = []
    for r in range(world):
        b = np.zeros(bucket_numel, dtype=dt)
        oracle.bucket_pack(grads_h[r], offsets, b, code)
        bufs.append(b)
    oracle.ring_allreduce(bufs, code, divisor)
    for r in range(world):
        oracle.bucket_unpack(grads_h[r], offsets, bufs[r], code)


def _oracle_view_hook(grads_h, offsets, bucket_numel, divisor, fp16=False):
    """Oracle steps of the bf16 (or fp16) hook on one bucket: pack the float32
    gradients, round, ring in the narrow type with divide, widen, unpack."""
    world = len(grads_h)
    rne, widen, code = ((oracle.fp16_rne, oracle.fp16_to_f32, oracle.F16) if fp16 else
                        (oracle.bf16_rne, oracle.bf16_to_f32, oracle.BF16))
    bufs = []
    for r in range(world):
        b = np.zeros(bucket_numel, dtype=np.float32)
        oracle.bucket_pack(grads_h[r], offsets, b, oracle.F32)
        bufs.append(rne(b))
    oracle.ring_allreduce(bufs, code, divisor)
    for r in range(world):
        oracle.bucket_unpack(grads_h[r], offsets, widen(bufs[r]), oracle.F32)


@pytest.mark.parametrize("kernel", VIEW_KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "hook", "hook16"])
@pytest.mark.parametrize("layout", ["boundaries", "pointers"])
def test_view_misaligned_chunks_or_pointers_match_oracle(dtype, layout, kernel):
    # a TMA-sized bucket (8 ranks) whose chunk boundaries are not 16-byte
    # aligned ("boundaries": every member 16-byte aligned in memory, the
    # chunk length odd), or whose members' pointers are not ("pointers":
    # members packed back to back at odd offsets in one arena).  The aligned
    # bodies go to the TMA kernel, the few elements around each boundary and
    # the misaligned members to the register kernel.
    # "hook" / "hook16": float32 gradients through the fused bf16 / fp16
    # compression hook
    hook = dtype if dtype in ("hook", "hook16") else None
    if hook:
        dtype = "f32"
    world = 8
    es = 2 if dtype == "bf16" else 4
    lanes = 16 // es
    if layout == "boundaries":
        numels = [lanes * 100_000, lanes * 1_000_001, 3 * lanes, lanes * 150_000]
    else:
        numels = [5, 1_000_003, 17, 1, 700_001, 6]
    total = sum(numels)
    offsets = list(np.cumsum([0] + numels[:-1]))
    if layout == "boundaries":
        assert (-(-total // world) * es) % 16 != 0
    host = []
    for r in range(world):
        xs = workloads.rank_vectors(1, total, "randn", std=1e-2, dtype=dtype, seed0=50 + r)[0]
        host.append(xs)
    if layout == "boundaries":
        dev = [[host[r][offsets[i]:offsets[i] + numels[i]].clone().to("cuda") for i in range(len(numels))]
               for r in range(world)]
    else:
        arenas = [h.to("cuda") for h in host]
        dev = [[arenas[r][offsets[i]:offsets[i] + numels[i]] for i in range(len(numels))] for r in range(world)]
        assert any(t.data_ptr() % 16 for t in dev[0])
    code = oracle.BF16 if dtype == "bf16" else oracle.F32
    for div in (world, 3):
        grads_h = [[f32_or_bits(t) for t in dev[r]] for r in range(world)]
        with _view_kernel(kernel):
            if hook == "hook":
                ddp.ddp_bucket_allreduce_view_bf16(dev, offsets, total, div)
            elif hook == "hook16":
                ddp.ddp_bucket_allreduce_view_fp16(dev, offsets, total, div)
            else:
                ddp.ddp_bucket_allreduce_view(dev, offsets, total, div)
        torch.cuda.synchronize()
        if hook:
            _oracle_view_hook(grads_h, offsets, total, div, fp16=hook == "hook16")
        else:
            _oracle_view(grads_h, offsets, total, code, div)
        for r in range(world):
            for i in range(len(numels)):
                assert_bits_equal(f32_or_bits(dev[r][i]), grads_h[r][i],
                                  f"{layout} {hook or dtype} {kernel} div={div} r{r} m{i}")
    assert ddp.ddp_device_status() == 0


@pytest.mark.parametrize("kernel", VIEW_KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "hook"])
def test_view_many_unaligned_boundaries_span_several_tma_launches(dtype, kernel):
    # 16 ranks, 5-7 buckets of odd sizes, every member its own aligned
    # allocation: the bodies go to the TMA view kernel, and the elements
    # around ~100 unaligned chunk boundaries and member ends (more than one
    # launch's edge table holds) are folded by its consumer warps, a member's
    # edges sometimes continuing in the next launch.  A few members are
    # shorter than 16 bytes (edges only).
    hook = dtype == "hook"
    if hook:
        dtype = "f32"
    world, first, cap = 16, 64 << 10, 2 << 20
    rng = np.random.default_rng(17)
    numels = [int(v) for v in rng.integers(20_000, 400_000, size=24)]
    numels[3], numels[11], numels[19] = 1, 3, 7
    es = 2 if dtype == "bf16" else 4
    code = oracle.BF16 if dtype == "bf16" else oracle.F32
    plan = ddp.ddp_plan_buckets(numels, code, first, cap)
    assert len(plan[2]) >= 4
    flat, grads_h = _host_grads(numels, world, dtype, seed0=57)
    offs = np.cumsum([0] + numels)
    dev = [[flat[r, int(offs[p]):int(offs[p + 1])].clone().to("cuda") for p in range(len(numels))]
           for r in range(world)]
    assert all(t.data_ptr() % 16 == 0 for t in dev[0])
    with _view_kernel(kernel):
        ddp.ddp_sync_buckets(dev, plan, None, algo=ddp.DDP_ALGO_BF16_HOOK_VIEW if hook else ddp.DDP_ALGO_VIEW)
    torch.cuda.synchronize()
    if hook:
        oracle.ddp_sync_bf16_hook(grads_h, first, cap)
    else:
        oracle.ddp_sync(grads_h, code, first, cap)
    for r in range(world):
        for p in range(len(numels)):
            assert_bits_equal(f32_or_bits(dev[r][p]), grads_h[r][p],
                              f"{'hook' if hook else dtype} {kernel} r{r} p{p}")
    assert ddp.ddp_device_status() == 0
    assert es in (2, 4)


@pytest.mark.parametrize("algo", ["fused", "staged", "hook"])
def test_one_scratch_buffer_shared_by_every_bucket(algo):
    # the bucket buffers may alias across buckets (one scratch per rank,
    # reused by every bucket): each bucket must then be packed, reduced and
    # unpacked before the next one is packed
    numels = _small_decoder()
    world, first, cap = 8, 4096, 40000
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, first, cap)
    assert len(plan[2]) > 2
    flat, grads_h = _host_grads(numels, world, "f32", seed0=41)
    g = flat.cuda()
    views = _device_views(g, numels)
    bdt = torch.bfloat16 if algo == "hook" else torch.float32
    scratch = [torch.empty(int(max(plan[2])), dtype=bdt, device="cuda") for _ in range(world)]
    bk = [[scratch[r][:int(n)] for n in plan[2]] for r in range(world)]
    code = {"fused": ddp.DDP_ALGO_FUSED, "staged": ddp.DDP_ALGO_STAGED, "hook": ddp.DDP_ALGO_BF16_HOOK}[algo]
    ddp.ddp_sync_buckets(views, plan, bk, algo=code)
    torch.cuda.synchronize()
    if algo == "hook":
        oracle.ddp_sync_bf16_hook(grads_h, first, cap)
    else:
        oracle.ddp_sync(grads_h, oracle.F32, first, cap)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"{algo} with one shared scratch buffer")


def test_python_usage_sequence_matches_oracle():
    # the binding's documented usage, written out here: plan, one view sync,
    # the same step overlapped through the reducer, and one bucket's fused
    # ring -- each result against the oracle
    numels = _small_decoder()
    world = 4
    flat, grads_h = _host_grads(numels, world, "f32", seed0=71)
    g = flat.cuda()
    grads = _device_views(g, numels)
    plan = ddp.ddp_plan_buckets([t.numel() for t in grads[0]], ddp.F32)
    ddp.ddp_sync_buckets(grads, plan, None, algo=ddp.DDP_ALGO_VIEW)
    torch.cuda.synchronize()
    oracle.ddp_sync(grads_h, oracle.F32)
    assert_bits_equal(f32_or_bits(g), np.stack([np.concatenate(grads_h[r]) for r in range(world)]), "view sync")

    flat2, grads2_h = _host_grads(numels, world, "f32", seed0=72)
    g2 = flat2.cuda()
    grads2 = _device_views(g2, numels)
    red = ddp.Reducer(grads2, plan, algo=ddp.DDP_ALGO_VIEW, comm_stream=torch.cuda.Stream())
    red.prepare()
    for p in reversed(range(len(numels))):
        red.mark_ready(p, torch.cuda.current_stream())
    red.finalize(torch.cuda.current_stream())
    torch.cuda.synchronize()
    red.close()
    oracle.ddp_sync(grads2_h, oracle.F32)
    assert_bits_equal(f32_or_bits(g2), np.stack([np.concatenate(grads2_h[r]) for r in range(world)]), "reducer")

    x = workloads.rank_vectors(world, 1000, "randn", seed0=3)
    xd = x.cuda()
    ddp.ring_allreduce_fused(xd, xd.shape[0])
    torch.cuda.synchronize()
    assert_bits_equal(f32_or_bits(xd), oracle_allreduce(x.numpy(), world), "one bucket")


def test_fp16_hook_view_overflow_and_subnormals_match_oracle():
    # binary16 range edges: sums past 65504 become infinity, values below
    # 2^-14 become subnormal or zero -- exactly as the oracle's binary16
    world, n = 4, 4096
    rng = np.random.default_rng(13)
    scale = np.where(np.arange(n) % 3 == 0, 3.0e4, np.where(np.arange(n) % 3 == 1, 1e-6, 1.0)).astype(np.float32)
    x = (rng.standard_normal((world, n)).astype(np.float32) * scale).astype(np.float32)
    big = np.arange(n) % 3 == 0
    x[:, big] = np.abs(x[:, big])      # one sign: infinities add up, never to NaN (NaN payloads are not compared)
    grads_h = [[x[r].copy()] for r in range(world)]
    g = torch.from_numpy(x.copy()).cuda()
    ddp.ddp_bucket_allreduce_view_fp16([[g[r]] for r in range(world)], [0], n, 0)
    torch.cuda.synchronize()
    oracle.ddp_sync_fp16_hook(grads_h, 1 << 40, 1 << 40, divisor=0)
    got = f32_or_bits(g)
    want = np.stack([grads_h[r][0] for r in range(world)])
    assert np.isinf(want).any() and (np.abs(want[want != 0]) < 6.2e-5).any()
    assert_bits_equal(got, want, "fp16 hook at the binary16 range edges")


@pytest.mark.parametrize("via", ["sync_buckets", "reducer"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "hook"])
def test_large_bucket_in_l2_pieces_matches_oracle(via, dtype):
    # a bucket of more than two L2-sized pieces (96 MiB of bucket over all
    # ranks each): members of odd sizes straddle the piece boundaries and
    # chunk boundaries; pack / ring / unpack run piece by piece and must give
    # the oracle's bits.  "hook": float32 gradients through the bf16
    # compression hook, whose bf16 bucket is cut into pieces the same way.
    hook = dtype == "hook"
    world = 4
    es = 2 if dtype in ("bf16", "hook") else 4
    piece = (96 << 20) // world // es // 1024 * 1024
    numels = [3, piece - 5, 7, piece + 11, 1001, piece // 3 + 17, 13]
    gdt = "f32" if hook else dtype
    code = ddp.BF16 if dtype == "bf16" else ddp.F32
    plan = ddp.ddp_plan_buckets(numels, code, 1 << 40, 1 << 40)
    assert len(plan[2]) == 1 and plan[2][0] > 2 * piece
    flat, grads_h = _host_grads(numels, world, gdt, seed0=81)
    g_storage, g = guarded_copy(flat)
    views = _device_views(g, numels)
    tdt = torch.bfloat16 if es == 2 else torch.float32
    bk = [[torch.empty(int(plan[2][0]), dtype=tdt, device="cuda")] for _ in range(world)]
    algo = ddp.DDP_ALGO_BF16_HOOK if hook else ddp.DDP_ALGO_FUSED
    if via == "sync_buckets":
        ddp.ddp_sync_buckets(views, plan, bk, algo=algo)
    else:
        red = ddp.Reducer(views, plan, bk, algo=algo, comm_stream=torch.cuda.Stream())
        for p in range(len(numels) - 1, -1, -1):
            red.mark_ready(p, torch.cuda.current_stream())
        red.finalize(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert_canaries(g_storage, f"pieces {dtype} via {via}")
    if hook:
        oracle.ddp_sync_bf16_hook(grads_h, 1 << 40, 1 << 40)
    else:
        oracle.ddp_sync(grads_h, code, 1 << 40, 1 << 40)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"pieces {dtype} via {via}")
    if via == "reducer":
        red.close()


@pytest.mark.parametrize("world", [3, 8])
@pytest.mark.parametrize("extra", [0, 1])
def test_pieces_switch_boundary_matches_oracle(world, extra):
    # a bucket of exactly 1.5 pieces runs whole; one element more runs in two
    # pieces (p and p/2 + 1).  At world 3 with the extra element the chunk
    # length is odd, so chunk boundaries inside the pieces are not 16-byte
    # aligned and the view kernel's edge path runs too.  Both must give the
    # oracle's bits.
    es = 4
    piece = max((96 << 20) // world // es // 1024 * 1024, 64 * 1024)
    total = piece + piece // 2 + extra
    numels = [12345, total - 12345]
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, 1 << 40, 1 << 40)
    assert list(plan[2]) == [total]
    flat, grads_h = _host_grads(numels, world, "f32", seed0=97)
    g = flat.cuda()
    views = _device_views(g, numels)
    bk = [[torch.empty(total, dtype=torch.float32, device="cuda")] for _ in range(world)]
    ddp.ddp_sync_buckets(views, plan, bk, algo=ddp.DDP_ALGO_FUSED)
    torch.cuda.synchronize()
    oracle.ddp_sync(grads_h, oracle.F32, 1 << 40, 1 << 40)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    assert_bits_equal(f32_or_bits(g), want, f"pieces boundary world={world} extra={extra}")
