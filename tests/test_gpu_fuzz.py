"""Seeded random parity: many small calls with random shapes, bit-exact vs the oracle.

Each case draws a world size, a bucket length, a dtype, a divisor, a start
offset inside 16-byte-aligned storage (so some calls take the element-wise
kernels), and a forced fused-kernel choice; it then runs one of the
allreduces or a view sync of a random member split, through the C ABI,
and compares every element with the oracle on the same input.  The rows
sit inside storage filled with a canary pattern, which must be intact
afterwards: no kernel may write outside the buffers it was given.
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


CANARY16 = 0x7FA5          # a bf16 NaN pattern that no kernel here produces
CANARY32 = 0x7FA5A5A5


def _rows_on_device(xh, shift):
    """Rank rows as views starting `shift` elements into aligned storage; the
    rest of the storage holds a canary pattern."""
    N, S = xh.shape
    bf = xh.dtype == np.uint16
    itype = torch.int16 if bf else torch.int32
    store = torch.full((N, S + 16), CANARY16 if bf else CANARY32, dtype=itype, device="cuda")
    store = store.view(torch.bfloat16 if bf else torch.float32)
    src = torch.from_numpy(xh.view(np.int16) if bf else xh)
    if bf:
        src = src.view(torch.bfloat16)
    rows = [store[r, shift:shift + S] for r in range(N)]
    for r in range(N):
        rows[r].copy_(src[r])
    return store, rows


def _canaries_intact(store, shift, S):
    bits = f32_or_bits(store)
    bits = bits.view(np.uint16) if bits.dtype == np.uint16 else bits.view(np.uint32)
    canary = CANARY16 if bits.dtype == np.uint16 else CANARY32
    outside = np.ones(bits.shape[1], dtype=bool)
    outside[shift:shift + S] = False
    return bool(np.all(bits[:, outside] == canary))


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
        what = f"case {block}/{case}: {op} N={N} S={S} {dtype} div={divisor} shift={shift} kind={kind}"
        assert_bits_equal(got, want, what)
        assert _canaries_intact(store, shift, S), "write outside the rank rows: " + what
        del store, rows
    assert ddp.ddp_device_status() == 0
