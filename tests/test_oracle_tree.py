"""Pins of the oracle's tree allreduce (binomial-tree reduce to rank 0,
divide, broadcast).

The pages name a tree-based allreduce as the latency-oriented alternative to
the ring for small messages ("DDP 与 Ring All-Reduce：梯度同步不是一次
AllReduce 就完事", sections 02 and 07, NCCL's Tree algorithm) without defining
it; the reading taken is the binomial tree.  Pins:
  * a hand-derived example with every intermediate state (N = 3);
  * bit-exact agreement with an independent recursive definition of the
    binomial pairwise sum, T(r, s) = T(r, s/2) (+) T(r + s/2, s/2);
  * an order pin only the pairwise association passes;
  * exact integer sums, identical ranks, traffic per rank, step count
    2 ceil(log2 N) (vs 2(N-1) for the ring).
"""
import math

import numpy as np
import pytest

import oracle


def test_hand_example_three_ranks_every_state():
    # x0 = [1, 2], x1 = [10, 20], x2 = [100, 200]
    base = np.array([[1, 2], [10, 20], [100, 200]], dtype=np.float32)
    states = {
        0: [[1, 2], [10, 20], [100, 200]],
        1: [[11, 22], [10, 20], [100, 200]],      # d = 1: rank 1 -> rank 0
        2: [[111, 222], [10, 20], [100, 200]],    # d = 2: rank 2 -> rank 0
        3: [[111, 222], [10, 20], [111, 222]],    # broadcast d = 2: rank 0 -> rank 2
        4: [[111, 222], [111, 222], [111, 222]],  # broadcast d = 1: rank 0 -> rank 1
    }
    for k, want in states.items():
        x = base.copy()
        oracle.tree_allreduce_2d(x, oracle.F32, 0, n_steps=k)
        np.testing.assert_array_equal(x, np.array(want, dtype=np.float32), err_msg=f"after {k} steps")
    x = base.copy()
    oracle.tree_allreduce_2d(x, oracle.F32, 3)
    np.testing.assert_array_equal(x, np.tile(np.array([37, 74], dtype=np.float32), (3, 1)))


def _pairwise(vals, r, size, n):
    """Binomial pairwise sum of ranks [r, min(r + size, n)), float32."""
    if size == 1:
        return np.float32(vals[r])
    half = size // 2
    left = _pairwise(vals, r, half, n)
    if r + half >= n:
        return left
    return np.float32(left + _pairwise(vals, r + half, half, n))


@pytest.mark.parametrize("N", list(range(1, 41)))
def test_matches_recursive_pairwise_definition(N):
    rng = np.random.default_rng(N)
    S = 9
    x = rng.standard_normal((N, S)).astype(np.float32)
    size = 1 << math.ceil(math.log2(N)) if N > 1 else 1
    want = np.array([_pairwise(x[:, i], 0, size, N) for i in range(S)], dtype=np.float32)
    y = oracle.tree_allreduce_2d(x.copy(), oracle.F32, 0)
    for r in range(N):
        np.testing.assert_array_equal(y[r], want)


def test_order_pin_pairwise_association():
    # (2^24 + 1) + (1 - 2^24) = 2^24 - 2^24 + 1 = 1 with the tree; the ring's
    # fold for this element gives 2, a left fold from rank 0 gives 0
    x = np.array([[2.0 ** 24], [1.0], [1.0], [-(2.0 ** 24)]], dtype=np.float32)
    assert np.all(oracle.tree_allreduce_2d(x.copy(), oracle.F32, 0) == 1.0)
    assert np.all(oracle.ring_allreduce_2d(x.copy(), oracle.F32, 0) == 2.0)


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 13, 64])
def test_exact_integers_identical_ranks_traffic_and_steps(N):
    rng = np.random.default_rng(100 + N)
    S = 23
    x = rng.integers(-50, 51, size=(N, S)).astype(np.float32)
    bufs = [x[r].copy() for r in range(N)]
    sent = oracle.tree_allreduce(bufs, oracle.F32, 0)
    exact = x.astype(np.float64).sum(0).astype(np.float32)
    for b in bufs:
        np.testing.assert_array_equal(b, exact)
    depth = math.ceil(math.log2(N)) if N > 1 else 0
    for r in range(N):
        # reduce: every rank but 0 sends its buffer once; broadcast: rank r sends
        # once per distance d with r % 2d == 0 and r + d < N
        bcast = sum(1 for k in range(depth) if r % (2 << k) == 0 and r + (1 << k) < N)
        assert sent[r] == S * ((1 if r else 0) + bcast)
    # step count: 2 ceil(log2 N) -- asking for one more step is refused
    with pytest.raises(ValueError):
        oracle.tree_allreduce([x[r].copy() for r in range(N)], oracle.F32, 0, 2 * depth + 1)
    if N == 64:
        assert 2 * depth == 12 and 2 * (N - 1) == 126


def test_bf16_tree_rounds_each_step():
    # bf16: (256 + 1) ties to 256, (256 + 256) = 512 exact -> with 4 ranks
    # [256, 1, 256, 0]: (256 + 1) -> 256, (256 + 0) = 256, 256 + 256 = 512
    f = np.array([[256.0], [1.0], [256.0], [0.0]], dtype=np.float32)
    h = oracle.bf16_rne(f)
    oracle.tree_allreduce_2d(h, oracle.BF16, 0)
    assert np.all(oracle.bf16_to_f32(h) == 512.0)
    # divide once at the root: 3 ranks of 1.0 / 3 rounds like the float32 quotient to bf16
    h = oracle.bf16_rne(np.ones((3, 1), dtype=np.float32))
    oracle.tree_allreduce_2d(h, oracle.BF16, 3)
    assert np.all(h == oracle.bf16_rne(np.array([1.0], dtype=np.float32))[0])
