"""Full-size ring allreduce parity: every element against the CPU oracle.

The method fixes the summation order of every element, so the ring's result
is one exact set of bits and the whole vector is compared, at every rank, at
the sizes the benchmarks run ("DDP 与 Ring-AllReduce", §1.3.2, shows every
element of every rank after every step; the fused kernel must reach the same
final state):
  * N = 8 ranks x 268,435,456 fp32 (1 GiB per rank), N(0, 1e-2^2), / 8 --
    the headline bucket -- through the fused ring (the kernel the size rule
    picks, and the vector kernel forced), the staged ring and the persistent
    ring;
  * the message-size sweep's largest points, 16 MiB and 256 MiB per rank of
    U[-1, 1) fp32, at N = 8 and N = 64;
  * bf16 at N = 16 with a ResNet-50-sized bucket (per-hop bf16 rounding);
  * 2 ranks of just over 2^31 elements each (indices past 32 bits).

Inputs are drawn on a CUDA generator (rank r from seed r) and snapshot to the
host before any kernel runs; the oracle runs on that snapshot.  Every run's
buffer sits between two canary regions, checked after the call.  Each case's
input and expected result are kept only while its tests run.
"""
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import (assert_canaries, assert_device_equals_host, guarded_copy, host_snapshot,
                      require_host_memory)

pytestmark = pytest.mark.gpu


def _persistent(x, divisor):
    st = ddp.ring_allreduce_persistent(x, divisor)
    torch.cuda.synchronize()
    assert int(st[0]) == 0, f"persistent ring status {int(st[0])}"


def _fused_vector(x, divisor):
    prev = ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_VECTOR)
    try:
        ddp.ring_allreduce_fused(x, divisor)
    finally:
        ddp.ddp_set_fused_kernel(prev)


def _fused_tma(x, divisor):
    prev = ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_TMA)
    try:
        ddp.ring_allreduce_fused(x, divisor)
    finally:
        ddp.ddp_set_fused_kernel(prev)


KERNELS = {"fused": ddp.ring_allreduce_fused, "fused_vector": _fused_vector, "fused_tma": _fused_tma,
           "staged": ddp.ring_allreduce_staged, "persistent": _persistent}

_case = {}


@pytest.fixture(scope="module", autouse=True)
def _release_full_size_buffers():
    yield
    _case.clear()
    torch.cuda.empty_cache()


def _inputs(N, S, kind, std, dtype):
    """(device input, host expected result, device float64 average) of one
    configuration, computed once while that configuration's tests run."""
    key = (N, S, kind, std, dtype)
    if key not in _case:
        _case.clear()
        torch.cuda.empty_cache()
        require_host_memory(N * S * (2 if dtype == "bf16" else 4), f"N={N} S={S}")
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        x0 = torch.empty((N, S), dtype=tdt, device="cuda")
        for r in range(N):
            v = (workloads.randn_f32(S, r, std, device="cuda") if kind == "randn"
                 else workloads.uniform_pm1_f32(S, r, device="cuda"))
            x0[r].copy_(v)
            del v
        ref64 = torch.zeros(S, dtype=torch.float64, device="cuda")
        for r in range(N):
            ref64 += x0[r].to(torch.float64)
        ref64 /= N
        torch.cuda.synchronize()
        want = host_snapshot(x0)
        oracle.ring_allreduce_2d(want, oracle.BF16 if dtype == "bf16" else oracle.F32, N)
        _case[key] = (x0, want, ref64)
    return _case[key]


def _check(kernel, N, S, kind, std, dtype):
    x0, want, ref64 = _inputs(N, S, kind, std, dtype)
    storage, x = guarded_copy(x0)
    KERNELS[kernel](x, N)
    torch.cuda.synchronize()
    assert_canaries(storage, f"{kernel} N={N} S={S}")
    assert_device_equals_host(x, want, f"{kernel} N={N} S={S} {dtype}")
    err = torch.linalg.vector_norm(x[0].to(torch.float64) - ref64) / torch.linalg.vector_norm(ref64)
    assert float(err) <= (2e-2 if dtype == "bf16" else 1e-5)
    del x, storage


@pytest.mark.parametrize("kernel", ["fused", "fused_vector", "staged", "persistent"])
def test_config_n8_one_gib_fp32_full(kernel):
    _check(kernel, 8, 1 << 28, "randn", 1e-2, "f32")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_sweep_n8_16_mib_full(kernel):
    _check(kernel, 8, (16 << 20) // 4, "uniform", 1.0, "f32")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_sweep_n8_256_mib_full(kernel):
    _check(kernel, 8, (256 << 20) // 4, "uniform", 1.0, "f32")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_sweep_n64_16_mib_full(kernel):
    _check(kernel, 64, (16 << 20) // 4, "uniform", 1.0, "f32")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_sweep_n64_256_mib_full(kernel):
    _check(kernel, 64, (256 << 20) // 4, "uniform", 1.0, "f32")


@pytest.mark.parametrize("kernel", ["fused", "staged", "persistent"])
def test_bf16_n16_resnet_sized_full(kernel):
    _check(kernel, 16, 25_557_032 // 2 + 3, "randn", 1e-2, "bf16")


@pytest.mark.parametrize("kernel,S", [("fused_tma", (1 << 31) + 8), ("fused_vector", (1 << 31) + 8),
                                      ("fused", (1 << 31) + 5)])
def test_more_than_2_31_elements_per_rank_full(kernel, S):
    # 2 ranks x just over 2^31 fp32 (8 GiB per rank): element, chunk and tile
    # indices past the 32-bit range, on the TMA kernel (16-byte chunks), the
    # vector kernel, and a ragged size (last vector done element-wise)
    _check(kernel, 2, S, "uniform", 1.0, "f32")
