"""Pins of the oracle's bucket plan, pack/unpack, no_sync accumulation and
bf16 rounding.

Bucket rule ("DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事",
section 03 "Bucket" and "Overlap"; section 05 step 2): parameters are taken
in reverse registration order, the first bucket is capped at 1 MiB and
every later one at 25 MiB ("MB" read as MiB, as that page does); a bucket is
closed once its bytes reach the cap.  The plan is pinned by a
characterisation that does not restate the loop: every parameter appears
once, offsets tile each bucket contiguously in reverse registration order,
each closed bucket reached its cap and was below it before its last member.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

MiB = 1024 * 1024


def check_plan_characterisation(numels, elem, first_cap, cap, b_of, off, bn):
    P = len(numels)
    K = len(bn)
    assert b_of.shape == (P,) and off.shape == (P,)
    if P == 0:
        assert K == 0
        return
    assert b_of.min() >= 0 and b_of.max() == K - 1
    # reverse registration order: walking p = P-1 .. 0 visits buckets 0,1,..
    # in order and offsets grow by the previous member's numel
    order = list(range(P - 1, -1, -1))
    expect_k, expect_off = 0, 0
    for p in order:
        if b_of[p] != expect_k:
            assert b_of[p] == expect_k + 1, "buckets must follow reverse registration order"
            assert expect_off == bn[expect_k], "bucket numel = sum of its members"
            expect_k, expect_off = expect_k + 1, 0
        assert off[p] == expect_off
        expect_off += numels[p]
    assert expect_k == K - 1 and expect_off == bn[K - 1]
    # caps: every bucket but the last reached its cap, and was below the cap
    # before its last member arrived
    for k in range(K):
        members = [p for p in order if b_of[p] == k]
        c = first_cap if k == 0 else cap
        total = sum(numels[p] for p in members) * elem
        before_last = total - numels[members[-1]] * elem
        assert before_last < c
        if k < K - 1:
            assert total >= c
    assert sum(bn) == sum(numels)


def test_plan_hand_example():
    # numels [10, 20, 30] fp32, first cap 100 B, cap 100 B.
    # reverse order: p2 (120 B >= 100) closes bucket 0 alone; p1 (80 B) then
    # p0 (+40 = 120 B) close bucket 1 with p1 at offset 0 and p0 at 20.
    b_of, off, bn = oracle.plan_buckets([10, 20, 30], 4, 100, 100)
    assert list(b_of) == [1, 1, 0]
    assert list(off) == [20, 0, 0]
    assert list(bn) == [30, 30]


def test_plan_hand_example_trailing_open_bucket():
    # caps 64 B; numels [1, 1, 16, 3]: p3 12 B, p2 +64 = 76 B -> close {p3,p2};
    # p1 4 B, p0 8 B -> left open, closed at the end.
    b_of, off, bn = oracle.plan_buckets([1, 1, 16, 3], 4, 64, 64)
    assert list(b_of) == [1, 1, 0, 0]
    assert list(off) == [1, 0, 3, 0]
    assert list(bn) == [19, 2]


def test_plan_first_bucket_uses_its_own_cap():
    # ten 1 KiB params, first cap 2 KiB, cap 4 KiB: bucket 0 takes 2, then 4, 4
    b_of, off, bn = oracle.plan_buckets([256] * 10, 4, 2048, 4096)
    assert list(bn) == [512, 1024, 1024]


def test_plan_empty_and_zero_sized():
    b_of, off, bn = oracle.plan_buckets([], 4, MiB, 25 * MiB)
    assert len(bn) == 0
    b_of, off, bn = oracle.plan_buckets([0, 5, 0], 4, 4, 4)
    check_plan_characterisation([0, 5, 0], 4, 4, 4, b_of, off, bn)


@pytest.mark.parametrize("seed", range(40))
def test_plan_characterisation_random(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 60))
    numels = [int(v) for v in rng.integers(0, 5000, size=P)]
    elem = int(rng.choice([2, 4]))
    first_cap = int(rng.integers(1, 20000))
    cap = int(rng.integers(1, 40000))
    b_of, off, bn = oracle.plan_buckets(numels, elem, first_cap, cap)
    check_plan_characterisation(numels, elem, first_cap, cap, b_of, off, bn)


def test_decoder_and_resnet_workload_totals():
    dec = workloads.param_numels(workloads.decoder_param_shapes())
    assert len(dec) == 292 and sum(dec) == 354_823_168 and sum(dec) * 4 == 1_419_292_672
    rn = workloads.param_numels(workloads.resnet50_param_shapes())
    assert len(rn) == 161 and sum(rn) == 25_557_032 and sum(rn) * 2 == 51_114_064


def test_decoder_plan_default_caps():
    dec = workloads.param_numels(workloads.decoder_param_shapes())
    b_of, off, bn = oracle.plan_buckets(dec, 4, MiB, 25 * MiB)
    check_plan_characterisation(dec, 4, MiB, 25 * MiB, b_of, off, bn)
    assert len(bn) == 37
    # bucket 0 is the last registered params (lnf, then block 23 from its end)
    assert b_of[len(dec) - 1] == 0 and b_of[len(dec) - 2] == 0
    assert b_of[0] == len(bn) - 1            # the embedding table goes last


@pytest.mark.parametrize("cap_mib,count", [(5, 9), (10, 6), (25, 3), (50, 2)])
def test_resnet_plan_cap_sweep(cap_mib, count):
    rn = workloads.param_numels(workloads.resnet50_param_shapes())
    b_of, off, bn = oracle.plan_buckets(rn, 2, MiB, cap_mib * MiB)
    check_plan_characterisation(rn, 2, MiB, cap_mib * MiB, b_of, off, bn)
    assert len(bn) == count
    # bucket 0 = fc weight + fc bias (the last two registered), 3.91 MiB
    assert bn[0] == 1000 * 2048 + 1000


def test_pack_is_reverse_concatenation_and_unpack_inverts():
    rng = np.random.default_rng(5)
    numels = [3, 0, 7, 1, 12, 5]
    for dtype, npdt in ((oracle.F32, np.float32), (oracle.BF16, np.uint16)):
        elem = 4 if dtype == oracle.F32 else 2
        b_of, off, bn = oracle.plan_buckets(numels, elem, 16, 40)
        grads = [rng.integers(0, 60000, size=n).astype(npdt) for n in numels]
        for k in range(len(bn)):
            members = oracle.bucket_members(b_of, off, k)
            buf = np.zeros(int(bn[k]), dtype=npdt)
            oracle.bucket_pack([grads[p] for p in members], [off[p] for p in members], buf, dtype)
            # bucket content = members concatenated in reverse registration order
            want = np.concatenate([grads[p] for p in sorted(members, reverse=True)]) if members else buf
            np.testing.assert_array_equal(buf, want)
            outs = [np.zeros_like(grads[p]) for p in members]
            oracle.bucket_unpack(outs, [off[p] for p in members], buf, dtype)
            for o, p in zip(outs, members):
                np.testing.assert_array_equal(o, grads[p])


def test_accumulate_small_integers_exact():
    rng = np.random.default_rng(11)
    g = [rng.integers(-100, 101, size=37).astype(np.float32) for _ in range(4)]
    acc = g[0].copy()
    for m in range(1, 4):
        oracle.accumulate(acc, g[m])
    np.testing.assert_array_equal(acc, np.sum(np.stack(g).astype(np.float64), axis=0).astype(np.float32))


def test_no_sync_then_sync_exact_on_integers():
    # 4 micro-batches, 2 ranks, 3 params, small integers: the accumulated,
    # averaged gradient is the exact mean over ranks of the sum over micro-batches
    rng = np.random.default_rng(12)
    N, M, numels = 2, 4, [5, 8, 3]
    micro = [[[rng.integers(-20, 21, size=n).astype(np.float32) for n in numels] for _ in range(N)]
             for _ in range(M)]
    acc = oracle.no_sync_then_sync(micro, oracle.F32, 16, 16)
    for p, n in enumerate(numels):
        tot = sum(micro[m][r][p].astype(np.float64) for m in range(M) for r in range(N))
        for r in range(N):
            np.testing.assert_array_equal(acc[r][p], (tot / N).astype(np.float32))


def test_bf16_rne_matches_torch_dense_sample():
    # every high half-word with a set of low half-words around the rounding
    # boundaries, plus random patterns; torch's float -> bfloat16 cast is an
    # independent implementation of round-to-nearest-even
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(0)
    pats = np.concatenate([pats, rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)])
    f = pats.view(np.float32)
    mine = oracle.bf16_rne(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    np.testing.assert_array_equal(mine[~nan], ref[~nan])
    # NaN stays NaN (exponent all ones, non-zero significand)
    m = mine[nan]
    assert np.all((m & 0x7F80) == 0x7F80) and np.all((m & 0x007F) != 0)


def test_bf16_widening_exact():
    h = np.arange(1 << 16, dtype=np.uint16)
    f = oracle.bf16_to_f32(h)
    t = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    same = (f.view(np.uint32) == t.view(np.uint32)) | (np.isnan(f) & np.isnan(t))
    assert np.all(same)


def test_bf16_hook_exact_on_small_integers_and_bounded_on_random():
    # small integers survive the rounding to bf16 and every hop exactly, and
    # the mean over 4 ranks is a multiple of 1/4: the hook must give it exactly
    rng = np.random.default_rng(21)
    N, numels = 4, [33, 7, 64, 5]
    grads = [[rng.integers(-8, 9, size=n).astype(np.float32) for n in numels] for _ in range(N)]
    exact = [sum(grads[r][p].astype(np.float64) for r in range(N)) / N for p in range(len(numels))]
    oracle.ddp_sync_bf16_hook(grads, 64, 128)
    for r in range(N):
        for p in range(len(numels)):
            np.testing.assert_array_equal(grads[r][p], exact[p].astype(np.float32))
    # random values: within the input rounding plus the per-hop bf16 bound
    u = 2.0 ** -8
    g = [[rng.standard_normal(n).astype(np.float32) * 1e-2 for n in numels] for _ in range(N)]
    x64 = [np.stack([g[r][p].astype(np.float64) for r in range(N)]) for p in range(len(numels))]
    oracle.ddp_sync_bf16_hook(g, 64, 128)
    for p in range(len(numels)):
        s_abs = np.abs(x64[p]).sum(0)
        bound = (u * s_abs + (N - 1) * u * s_abs * (1 + u)) / N + u * np.abs(x64[p].sum(0) / N) * 1.01
        assert np.all(np.abs(g[0][p].astype(np.float64) - x64[p].sum(0) / N) <= bound + 1e-12)

