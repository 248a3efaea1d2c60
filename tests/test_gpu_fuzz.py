"""Seeded random parity: many small calls with random shapes, bit-exact vs the oracle.

Each case draws a world size, a bucket length, a dtype, a divisor, a start
offset inside 16-byte-aligned storage (so some calls take the element-wise
kernels), and a forced fused-kernel choice; it then runs one of the
allreduces or a view sync of a random member split, through the C ABI,
and compares every element with the oracle on the same input.
"""
import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import assert_bits_equal, f32_or_bits

pytestmark = pytest.mark.gpu

KINDS = [ddp.DDP_FUSED_AUTO, ddp.DDP_FUSED_VECTOR, ddp.DDP_FUSED_GROUP, ddp.DDP_FUSED_TMA]


def _rows_on_device(xh, shift):
    """Rank rows as views starting `shift` elements into aligned storage."""
    N, S = xh.shape
    tdt = torch.bfloat16 if xh.dtype == np.uint16 else torch.float32
    store = torch.zeros((N, S + 16), dtype=tdt, device="cuda")
    src = torch.from_numpy(xh.view(np.int16) if xh.dtype == np.uint16 else xh)
    if xh.dtype == np.uint16:
        src = src.view(torch.bfloat16)
    rows = [store[r, shift:shift + S] for r in range(N)]
    for r in range(N):
        rows[r].copy_(src[r])
    return store, rows


def _oracle(op, xh, divisor):
    y = np.ascontiguousarray(xh).copy()
    code = oracle.BF16 if y.dtype == np.uint16 else oracle.F32
    if op == "tree":
        oracle.tree_allreduce_2d(y, code, divisor)
    else:                       # ring and view (the view's result is the bucket's ring result)
        oracle.ring_allreduce_2d(y, code, divisor)
    return y


@pytest.mark.parametrize("block", range(4))
def test_random_calls_match_oracle(block):
    rng = np.random.default_rng(1000 + block)
    for case in range(50):
        op = rng.choice(["ring_fused", "ring_staged", "tree", "view"])
        N = int(rng.integers(1, 65 if op == "tree" else 41))
        S = int(rng.choice([rng.integers(0, 64), rng.integers(64, 5000), rng.integers(5000, 300_000)]))
        dtype = "bf16" if rng.random() < 0.4 else "f32"
        divisor = int(rng.choice([0, 1, N, 3, 16]))
        shift = int(rng.choice([0, 0, 0, 1, 3]))
        kind = int(rng.choice(KINDS))
        xh = f32_or_bits(workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype,
                                                seed0=int(rng.integers(0, 1 << 20))))
        want = _oracle("tree" if op == "tree" else "ring", xh, divisor)
        store, rows = _rows_on_device(xh, shift)
        prev = ddp.ddp_set_fused_kernel(kind)
        try:
            if op == "ring_fused":
                ddp.ring_allreduce_fused(rows, divisor)
            elif op == "ring_staged":
                ddp.ring_allreduce_staged(rows, divisor)
            elif op == "tree":
                ddp.tree_allreduce_fused(rows, divisor)
            else:
                # a random split of the bucket into members, each a view of its rank row
                cuts = sorted(set(int(c) for c in rng.integers(0, S + 1, size=int(rng.integers(0, 6)))))
                bounds = [0] + cuts + [S]
                offsets = [a for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
                numels = [b - a for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
                views = [[rows[r][o:o + n] for o, n in zip(offsets, numels)] for r in range(N)]
                if numels:
                    ddp.ddp_bucket_allreduce_view(views, offsets, S, divisor)
        finally:
            ddp.ddp_set_fused_kernel(prev)
        torch.cuda.synchronize()
        got = np.stack([f32_or_bits(rows[r]) for r in range(N)]) if N else np.zeros((0, S))
        assert_bits_equal(got, want, f"case {block}/{case}: {op} N={N} S={S} {dtype} div={divisor} "
                                     f"shift={shift} kind={kind}")
        del store, rows
    assert ddp.ddp_device_status() == 0
