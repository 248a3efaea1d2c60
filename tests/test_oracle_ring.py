"""Pins of the oracle's ring allreduce against facts fixed outside the oracle.

Each pin comes from the pages or from mathematics, never from the oracle
itself:
  * the worked example's printed states ("DDP 与 Ring-AllReduce", §1.3.2,
    transcribed in tests/golden/ring_3x6_example.txt);
  * the per-chunk summation order the example implies (chunk j starts at
    rank j+1 and ends at rank j), pinned by values for which only that
    association gives the right float32 / bf16 answer;
  * an exact float64 sum on small integer inputs (every order is exact);
  * the classical recursive-summation error bound on random inputs;
  * the ring's traffic accounting ("DDP 与 Ring All-Reduce：梯度同步不是一次
    AllReduce 就完事" section 04; "DDP 与 Ring-AllReduce" §1.3.3):
    2(N-1) steps, 2(N-1)/N * S elements sent per rank, +12.5 % and x9 steps
    from N = 8 to N = 64;
  * special cases (one rank, empty vector, equal inputs).
"""
import os
import re

import numpy as np
import torch
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_3x6_example.txt")


# --------------------------------------------------------------------------
# 1. The worked example, every intermediate state
# --------------------------------------------------------------------------

def _example_inputs():
    # a_k = k+1, b_k = 10(k+1), c_k = 100(k+1): every sum is exact and each
    # decimal digit of a result names the ranks that contributed to it.
    k = np.arange(6, dtype=np.float32)
    return [(k + 1).astype(np.float32), (10 * (k + 1)).astype(np.float32), (100 * (k + 1)).astype(np.float32)]


def _golden_states():
    states = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, rest = line.split(" ", 2)[:2], line.split(" ", 2)[2]
            state, gpu = head[0], int(head[1])
            chunks = [c.strip() for c in rest.split("|")]
            assert len(chunks) == 3
            states.setdefault(state, {})[gpu] = chunks
    return states


def _eval_chunk(expr, j, inputs):
    """Evaluate e.g. 'A1+C1' or 'S2' to the two values of that chunk."""
    names = {"A": inputs[0], "B": inputs[1], "C": inputs[2]}
    total = np.zeros(2, dtype=np.float64)
    for term in expr.split("+"):
        m = re.fullmatch(r"([ABCS])(\d)", term.strip())
        assert m, term
        letter, idx = m.group(1), int(m.group(2))
        assert idx == j, f"term {term} placed in chunk {j}"
        if letter == "S":
            for v in inputs:
                total += v[2 * idx: 2 * idx + 2]
        else:
            total += names[letter][2 * idx: 2 * idx + 2]
    return total


def test_golden_fixture_shape():
    st = _golden_states()
    assert list(st) == ["init", "rs1", "rs2", "ag1", "ag2"]
    assert all(sorted(v) == [0, 1, 2] for v in st.values())


@pytest.mark.parametrize("k,state", [(0, "init"), (1, "rs1"), (2, "rs2"), (3, "ag1"), (4, "ag2")])
def test_worked_example_state(k, state):
    inputs = _example_inputs()
    bufs = [v.copy() for v in inputs]
    oracle.ring_allreduce(bufs, oracle.F32, divisor=0, n_steps=k)
    gold = _golden_states()[state]
    for g in range(3):
        want = np.concatenate([_eval_chunk(gold[g][j], j, inputs) for j in range(3)]).astype(np.float32)
        np.testing.assert_array_equal(bufs[g], want, err_msg=f"{state} GPU{g}")


def test_worked_example_final_average():
    bufs = [v.copy() for v in _example_inputs()]
    sent = oracle.ring_allreduce(bufs, oracle.F32, divisor=3)
    want = (37 * (np.arange(6) + 1)).astype(np.float32)      # 111(k+1) / 3
    for b in bufs:
        np.testing.assert_array_equal(b, want)
    # 2(N-1)/N * S = 4/3 * 6 = 8 elements sent by every rank
    assert list(sent) == [8, 8, 8]


# --------------------------------------------------------------------------
# 2. Association order: chunk j is folded starting at rank j+1
# --------------------------------------------------------------------------

def test_order_pin_fp32_three_ranks():
    # chunk j holds 2^24 on rank j+1, 1 on rank j+2 and -2^24 on rank j:
    # (2^24 + 1) rounds back to 2^24 (tie to even), so only the fold that
    # starts at rank j+1 gives 0; starting at j+2 or at j gives 1.
    N = 3
    x = np.zeros((N, N), dtype=np.float32)
    for j in range(N):
        x[(j + 1) % N, j] = 2.0 ** 24
        x[(j + 2) % N, j] = 1.0
        x[j, j] = -(2.0 ** 24)
    for start, want in ((1, 0.0), (2, 1.0), (0, 1.0)):
        got = np.float32(np.float32(np.float32(x[(0 + start) % N, 0]) + x[(1 + start) % N, 0]) + x[(2 + start) % N, 0])
        assert got == want
    oracle.ring_allreduce_2d(x, oracle.F32)
    assert np.all(x == 0.0), x


def test_order_pin_fp32_direction_four_ranks():
    # With N = 4 a ring running the other way (rank r sends to r-1) folds
    # chunk j as x[j-1], x[j-2], x[j-3], x[j] and would give 2 here; the page's
    # direction (GPU0 -> GPU1 -> GPU2 -> GPU0) gives 0.
    N = 4
    x = np.zeros((N, N), dtype=np.float32)
    for j in range(N):
        x[(j + 1) % N, j] = 2.0 ** 24
        x[(j + 2) % N, j] = 1.0
        x[(j + 3) % N, j] = 1.0
        x[j, j] = -(2.0 ** 24)
    oracle.ring_allreduce_2d(x, oracle.F32)
    assert np.all(x == 0.0), x


def test_order_pin_bf16():
    # bf16 keeps 8 significant bits: 256 + 1 = 257 is a tie between 256 and
    # 258 and rounds to 256, so again only the fold from rank j+1 gives 0.
    N = 3
    f = np.zeros((N, N), dtype=np.float32)
    for j in range(N):
        f[(j + 1) % N, j] = 256.0
        f[(j + 2) % N, j] = 1.0
        f[j, j] = -256.0
    h = oracle.bf16_rne(f)
    oracle.ring_allreduce_2d(h, oracle.BF16)
    assert np.all(oracle.bf16_to_f32(h) == 0.0)


def test_bf16_rounds_to_nearest_even_after_every_hop():
    # chunk j holds 256 on rank j+1, 3 on rank j+2, -256 on rank j.  The first
    # hop gives 259, a tie between the bf16 neighbours 258 and 260, which
    # rounds to 260 (even significand); the second hop gives 260 - 256 = 4.
    # Rounding once at the end would give 3, truncating each hop 258 - 256 = 2.
    N = 3
    f = np.zeros((N, N), dtype=np.float32)
    for j in range(N):
        f[(j + 1) % N, j] = 256.0
        f[(j + 2) % N, j] = 3.0
        f[j, j] = -256.0
    h = oracle.bf16_rne(f)
    oracle.ring_allreduce_2d(h, oracle.BF16)
    assert np.all(oracle.bf16_to_f32(h) == 4.0), oracle.bf16_to_f32(h)
    # a non-tie: 256 + 1.5 = 257.5 is nearer 258 than 256 (truncation: 256)
    f2 = np.zeros((2, 2), dtype=np.float32)
    f2[1, 0], f2[0, 0] = 256.0, 1.5       # chunk 0 starts at rank 1
    f2[0, 1], f2[1, 1] = 256.0, 1.5       # chunk 1 starts at rank 0
    h2 = oracle.bf16_rne(f2)
    oracle.ring_allreduce_2d(h2, oracle.BF16)
    assert np.all(oracle.bf16_to_f32(h2) == 258.0)


def test_order_pin_with_chunks_longer_than_one():
    # Same pin, S = 5 with N = 3 (chunks of 2, 2, 1): checks the ceil(S/N)
    # chunk boundaries as well as the start rank of every element.
    N, S = 3, 5
    c = -(-S // N)
    x = np.zeros((N, S), dtype=np.float32)
    for i in range(S):
        j = i // c
        x[(j + 1) % N, i] = 2.0 ** 24
        x[(j + 2) % N, i] = 1.0
        x[j, i] = -(2.0 ** 24)
    oracle.ring_allreduce_2d(x, oracle.F32)
    assert np.all(x == 0.0), x


# --------------------------------------------------------------------------
# 3. Brute force against float64 on tiny inputs
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N", list(range(1, 10)))
def test_integer_inputs_equal_exact_sum(N):
    rng = np.random.default_rng(1000 + N)
    for S in list(range(0, 71)):
        x = rng.integers(-50, 51, size=(N, S)).astype(np.float32)
        exact = x.astype(np.float64).sum(axis=0)
        y = oracle.ring_allreduce_2d(x.copy(), oracle.F32, divisor=0)
        for r in range(N):
            np.testing.assert_array_equal(y[r], exact.astype(np.float32))
        # the average: exact sum / N rounded once to float32 (the float64
        # quotient rounded to float32 is correctly rounded: 53 >= 2*24+2)
        z = oracle.ring_allreduce_2d(x.copy(), oracle.F32, divisor=N)
        want = (exact / N).astype(np.float32) if N > 1 else exact.astype(np.float32)
        for r in range(N):
            np.testing.assert_array_equal(z[r], want)


@pytest.mark.parametrize("N", [2, 3, 5, 8, 9])
def test_random_inputs_within_summation_bound(N):
    rng = np.random.default_rng(7 + N)
    u = 2.0 ** -24
    for S in (1, 7, 31, 64, 70):
        x = rng.standard_normal((N, S)).astype(np.float32)
        x64 = x.astype(np.float64)
        s64 = x64.sum(axis=0)
        bound_sum = (N - 1) * u * np.abs(x64).sum(axis=0) * (1 + 1e-12)
        y = oracle.ring_allreduce_2d(x.copy(), oracle.F32, divisor=0)
        assert np.all(np.abs(y[0].astype(np.float64) - s64) <= bound_sum)
        z = oracle.ring_allreduce_2d(x.copy(), oracle.F32, divisor=N)
        bound_avg = bound_sum / N + u * np.abs(s64 / N) * 1.000001
        assert np.all(np.abs(z[0].astype(np.float64) - s64 / N) <= bound_avg + 1e-45)


@pytest.mark.parametrize("N", [2, 4, 16])
def test_bf16_random_within_bound_and_small_integers_exact(N):
    rng = np.random.default_rng(99 + N)
    u = 2.0 ** -8
    S = 67
    x = rng.standard_normal((N, S)).astype(np.float32) * 1e-2
    h = oracle.bf16_rne(x)
    xf = oracle.bf16_to_f32(h).astype(np.float64)
    s64 = xf.sum(axis=0)
    y = oracle.ring_allreduce_2d(h.copy(), oracle.BF16, divisor=N)
    yf = oracle.bf16_to_f32(y[0]).astype(np.float64)
    bound = ((N - 1) * u * np.abs(xf).sum(axis=0)) / N + u * np.abs(s64 / N) * 1.0001
    assert np.all(np.abs(yf - s64 / N) <= bound)
    # small integers: sums stay below 256 in magnitude, so bf16 holds them exactly
    xi = rng.integers(-8, 9, size=(N, S)).astype(np.float32)
    hi = oracle.bf16_rne(xi)
    yi = oracle.ring_allreduce_2d(hi.copy(), oracle.BF16, divisor=0)
    np.testing.assert_array_equal(oracle.bf16_to_f32(yi[N - 1]), xi.sum(axis=0).astype(np.float32))


# --------------------------------------------------------------------------
# 4. Invariants and closed forms of the ring
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,S", [(1, 5), (2, 7), (3, 6), (4, 1), (5, 3), (8, 64), (7, 100), (9, 70)])
def test_all_ranks_identical_and_sent_volume(N, S):
    rng = np.random.default_rng(N * 100 + S)
    x = rng.standard_normal((N, S)).astype(np.float32)
    bufs = [x[r].copy() for r in range(N)]
    sent = oracle.ring_allreduce(bufs, oracle.F32, divisor=N)
    for r in range(1, N):
        assert bufs[r].tobytes() == bufs[0].tobytes()
    # reduce-scatter step s sends chunk r-s (s = 1..N-1): every chunk but r;
    # all-gather step t sends chunk r-t+1 (t = 1..N-1): every chunk but r+1.
    # So rank r sends (S - |chunk r|) + (S - |chunk r+1|) elements, which is
    # 2(N-1)/N * S when N divides S.
    c = -(-S // N)

    def clen(j):
        return min((j + 1) * c, S) - min(j * c, S)

    for r in range(N):
        assert sent[r] == (S - clen(r)) + (S - clen((r + 1) % N))
    assert sent.sum() == 2 * (N - 1) * S
    if S % N == 0:
        assert all(s * N == 2 * (N - 1) * S for s in sent)


def test_step_count_is_two_phases_of_n_minus_one():
    # asking for more than 2(N-1) steps is refused; 2(N-1) completes the sum
    for N in (2, 3, 8):
        x = np.ones((N, 2 * N), dtype=np.float32)
        with pytest.raises(ValueError):
            oracle.ring_allreduce([x[r].copy() for r in range(N)], oracle.F32, 0, 2 * (N - 1) + 1)
        bufs = [x[r].copy() for r in range(N)]
        oracle.ring_allreduce(bufs, oracle.F32, 0, 2 * (N - 1))
        assert all(np.all(b == N) for b in bufs)
        # one step short of the end, some rank still misses a chunk
        bufs = [x[r].copy() for r in range(N)]
        oracle.ring_allreduce(bufs, oracle.F32, 0, 2 * (N - 1) - 1)
        assert not all(np.all(b == N) for b in bufs)


def test_n8_to_n64_closed_forms():
    # section 04 of the first page: from N=8 to N=64 the per-rank volume grows
    # from 1.75 S to 1.96875 S (+12.5 %) and the step count from 14 to 126 (x9)
    S = 64 * 8
    vol = {}
    for N in (8, 64):
        x = np.ones((N, S), dtype=np.float32)
        sent = oracle.ring_allreduce([x[r].copy() for r in range(N)], oracle.F32, 0)
        vol[N] = sent[0] / S
    assert vol[8] == 1.75 and vol[64] == 1.96875
    assert abs(vol[64] / vol[8] - 1.125) < 1e-12
    assert (2 * (64 - 1)) / (2 * (8 - 1)) == 9


# --------------------------------------------------------------------------
# 5. Special cases
# --------------------------------------------------------------------------

def test_single_rank_is_identity_or_plain_divide():
    x = np.random.default_rng(3).standard_normal(33).astype(np.float32)
    y = x.copy()
    sent = oracle.ring_allreduce([y], oracle.F32, divisor=0)
    np.testing.assert_array_equal(y, x)
    assert sent[0] == 0
    y = x.copy()
    oracle.ring_allreduce([y], oracle.F32, divisor=3)
    np.testing.assert_array_equal(y, (x / np.float32(3)).astype(np.float32))


def test_empty_vector_is_noop():
    bufs = [np.zeros(0, dtype=np.float32) for _ in range(4)]
    sent = oracle.ring_allreduce(bufs, oracle.F32, divisor=4)
    assert list(sent) == [0, 0, 0, 0]


def test_equal_inputs_give_n_times_value():
    for N in (2, 3, 4, 7):
        v = np.float32(0.375)
        x = np.full((N, 11), v, dtype=np.float32)
        oracle.ring_allreduce_2d(x, oracle.F32, 0)
        assert np.all(x == np.float32(N * 0.375))


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.ring_allreduce([np.zeros(3, np.float32)], oracle.F32, divisor=-1)


def test_openmp_build_gives_identical_bits():
    # the multi-core timing build runs the ranks of each half-step on threads;
    # every element sees the same operations in the same order
    import subprocess
    try:
        oracle.build(openmp=True)
    except (subprocess.CalledProcessError, OSError):
        pytest.skip("no OpenMP in this compiler")
    for N, S, dtype in ((3, 6, oracle.F32), (8, 100_003, oracle.F32), (5, 77_777, oracle.BF16), (16, 4099, oracle.F32)):
        x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype="bf16" if dtype == oracle.BF16 else "f32")
        xh = x.view(torch.int16).numpy().view(np.uint16).copy() if dtype == oracle.BF16 else x.numpy().copy()
        a = oracle.ring_allreduce_2d(xh.copy(), dtype, N)
        b = oracle.ring_allreduce_2d_openmp(xh.copy(), dtype, N)
        assert np.array_equal(a.view(np.uint16 if dtype == oracle.BF16 else np.uint32),
                              b.view(np.uint16 if dtype == oracle.BF16 else np.uint32)), (N, S)
