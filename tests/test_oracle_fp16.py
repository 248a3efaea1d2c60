"""Pins for the oracle's IEEE binary16 arithmetic (the fp16 compression hook).

The fp16 hook rounds every gradient to binary16, reduces in a binary16 ring
with one rounding per hop, and widens the result back to float32 ("Day 17 ·
梯度的集体行动", reading list: DDP communication hooks, fp16/bf16
compression).  The oracle's rounding is written from the IEEE definition;
these tests pin it to torch's float -> half cast and to hand-computed cases.
"""
import numpy as np
import torch

import oracle
import workloads


def _torch_half_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float16).view(torch.int16) \
        .numpy().view(np.uint16)


def _same_or_both_nan(mine, ref):
    mine_nan = (mine & 0x7C00) == 0x7C00
    mine_nan &= (mine & 0x3FF) != 0
    ref_nan = ((ref & 0x7C00) == 0x7C00) & ((ref & 0x3FF) != 0)
    assert np.array_equal(mine_nan, ref_nan)
    assert np.array_equal(mine[~mine_nan], ref[~ref_nan])


def test_fp16_rne_matches_torch_on_random_bit_patterns():
    bits = np.random.default_rng(0).integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    _same_or_both_nan(oracle.fp16_rne(x), _torch_half_bits(x))


def test_fp16_rne_matches_torch_at_every_rounding_boundary():
    # every binary16 value, the float32 neighbours of it, and the float32
    # values around each midpoint between consecutive binary16 values
    h = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)           # finite non-negative halves
    v = oracle.fp16_to_f32(h).astype(np.float64)
    nxt = np.append(v[1:], 65520.0)                                       # 65520: where rounding reaches inf
    mid = (v + nxt) / 2
    cand = np.concatenate([v, mid]).astype(np.float32)
    cb = cand.view(np.uint32)
    cand = np.concatenate([cb - 1, cb, cb + 1]).view(np.float32)
    cand = np.concatenate([cand, -cand])
    _same_or_both_nan(oracle.fp16_rne(cand), _torch_half_bits(cand))
    assert oracle.fp16_rne(np.float32([65519.99, 65520.0, 2.0 ** -25, 2.0 ** -25 * 1.0001])).tolist() == \
        [0x7BFF, 0x7C00, 0x0000, 0x0001]


def test_fp16_widening_is_exact_for_every_pattern():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.fp16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.float16).float().numpy()
    both_nan = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine.view(np.uint32)[~both_nan], ref.view(np.uint32)[~both_nan])


def test_fp16_ring_rounds_every_hop_in_ring_order():
    # chunk j is folded from rank j+1: (2048 + 1) ties to 2048 in binary16,
    # + 1 ties to 2048 again; exact or end-rounded summation would give 2050,
    # any other start rank 2050 as well (1 + 1 = 2, + 2048 = 2050)
    N = 3
    x = np.zeros((N, N), dtype=np.float32)
    for j in range(N):
        x[(j + 1) % N, j], x[(j + 2) % N, j], x[j, j] = 2048.0, 1.0, 1.0
    bufs = [oracle.fp16_rne(x[r]) for r in range(N)]
    oracle.ring_allreduce(bufs, oracle.F16, 0)
    for r in range(N):
        assert oracle.fp16_to_f32(bufs[r]).tolist() == [2048.0] * N


def test_fp16_hook_on_small_integers_is_the_rounded_average():
    # integers up to 2^11 are exact in binary16, so every hop is exact; the
    # result is the float32 average rounded once to binary16
    world, numels = 4, [5, 300, 17, 1000]
    flat = workloads.rank_vectors(world, sum(numels), "int", seed0=2).numpy()
    offs = np.cumsum([0] + numels)
    grads = [[flat[r, offs[p]:offs[p + 1]].copy() for p in range(len(numels))] for r in range(world)]
    oracle.ddp_sync_fp16_hook(grads, 1 << 40, 1 << 40)
    want = oracle.fp16_to_f32(oracle.fp16_rne((flat.astype(np.float64).sum(0) / world).astype(np.float32)))
    for r in range(world):
        np.testing.assert_array_equal(np.concatenate(grads[r]), want)
