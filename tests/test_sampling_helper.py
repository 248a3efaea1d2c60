"""The sampled-expectation helper used by the large GPU parity tests must give
exactly the full oracle's values at the sampled elements (CPU only)."""
import numpy as np
import torch
import pytest

import oracle
import workloads
from gpu_util import chunk_index, oracle_allreduce, sample_indices, sampled_expected


@pytest.mark.parametrize("N,S,dtype,div", [(2, 1001, "f32", 2), (5, 10_007, "f32", 5), (8, 65_536, "f32", 8),
                                           (3, 999, "bf16", 3), (16, 40_009, "bf16", 16), (7, 13, "f32", 0)])
def test_sampled_expected_equals_full_oracle(N, S, dtype, div):
    x = workloads.rank_vectors(N, S, "randn", std=1e-2, dtype=dtype, seed0=N)
    xh = x.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else x.numpy()
    full = oracle_allreduce(xh, div)
    idx = sample_indices(S, N, 500, seed=1)
    got = sampled_expected(xh[:, idx].copy(), chunk_index(idx, S, N), N, div)
    assert np.array_equal(got.view(np.uint16 if dtype == "bf16" else np.uint32),
                          full[:, idx].view(np.uint16 if dtype == "bf16" else np.uint32))


def test_sample_indices_cover_every_chunk_boundary():
    S, N = 1000, 7
    idx = set(sample_indices(S, N, 0).tolist())
    c = -(-S // N)
    for j in range(N):
        assert j * c in idx and min((j + 1) * c, S) - 1 in idx


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_full_size_compare_helpers_find_a_planted_difference(dtype):
    # the chunked comparison used by the full-size GPU parity tests, run on
    # CPU tensors: equal data passes, one changed bit anywhere is found
    from gpu_util import assert_device_equals_host, host_snapshot
    x = workloads.rank_vectors(3, 10_001, "randn", dtype=dtype, seed0=5)
    h = host_snapshot(x)
    assert h.dtype == (np.uint16 if dtype == "bf16" else np.float32)
    assert_device_equals_host(x, h, "equal", piece=1000)
    for r, i in ((0, 0), (2, 10_000), (1, 4_321)):
        bad = h.copy()
        v = bad.view(np.uint16 if dtype == "bf16" else np.uint32)
        v[r, i] ^= 1
        with pytest.raises(AssertionError, match=f"rank {r}: 1 mismatches .* first at {i}"):
            assert_device_equals_host(x, bad, "planted", piece=1000)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_canary_guards_keep_alignment_and_catch_overwrites(dtype):
    # the guards the GPU parity tests put around their buffers, on CPU tensors
    from gpu_util import CANARY_BYTES, assert_canaries, guarded
    storage, view = guarded((3, 1001), dtype, device="cpu")
    assert view.data_ptr() - storage.data_ptr() == CANARY_BYTES and CANARY_BYTES % 512 == 0
    view.fill_(1.0)
    assert_canaries(storage, "untouched")
    iv = torch.int16 if dtype == torch.bfloat16 else torch.int32
    pad = CANARY_BYTES // view.element_size()
    for where in (0, pad - 1, storage.numel() - pad, storage.numel() - 1):
        bad = storage.clone()
        bad.view(iv)[where] = 0
        with pytest.raises(AssertionError, match="guard elements"):
            assert_canaries(bad, "planted")
