"""Full-size DDP step parity on the 355M-parameter decoder: every gradient
element of every rank against the CPU oracle.

Workload: the 24-layer decoder's 292 gradients (354,823,168 fp32 per rank),
N = 8 ranks, rank r's gradients N(0, 1e-2^2) from seed r on a CUDA generator,
snapshot to the host before any kernel runs.  Expected values come from the
oracle alone -- its own bucket plan (reverse registration order, 1 MiB first
bucket, 25 MiB cap; 37 buckets), its pack, its ring and its unpack
(``oracle.ddp_sync``; the hooks' and no_sync's compositions likewise) -- and
the library runs the step with its own plan through ddp_sync_buckets or the
reducer:
  * pack + fused ring + unpack (large buckets in L2-sized pieces), pack +
    staged ring + unpack, and the fused view;
  * the reducer, buckets launched as backward would make them ready;
  * the bf16 compression hook, unfused and fused, and the fused fp16 hook;
  * no_sync: 4 micro-batches (rank r's m-th from seed r + 8m) accumulated
    locally, then one sync.
The gradient arena and every bucket buffer sit between canary regions,
checked after each step.
"""
import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import (assert_canaries, assert_device_equals_host, guarded, guarded_copy, host_snapshot,
                      require_host_memory)

pytestmark = pytest.mark.gpu
MiB = 1 << 20
WORLD = 8
NUMELS = workloads.param_numels(workloads.decoder_param_shapes())
TOTAL = sum(NUMELS)
OFFS = np.cumsum([0] + NUMELS)
MICRO = 4

_case = {}


@pytest.fixture(scope="module", autouse=True)
def _release_full_size_buffers():
    yield
    _case.clear()
    torch.cuda.empty_cache()


def _draw(m):
    """Micro-batch m of every rank, on the device: [WORLD, TOTAL] fp32."""
    g = torch.empty((WORLD, TOTAL), dtype=torch.float32, device="cuda")
    for r in range(WORLD):
        g[r].copy_(workloads.randn_f32(TOTAL, workloads.microbatch_seed(r, WORLD, m), 1e-2, device="cuda"))
    return g


def _views(flat):
    return [[flat[r, int(OFFS[p]):int(OFFS[p + 1])] for p in range(len(NUMELS))] for r in range(flat.shape[0])]


def _expected(kind):
    """(device micro-batch 0, host expected gradients) for one kind of step,
    computed once while that kind's tests run."""
    if kind not in _case:
        _case.clear()
        torch.cuda.empty_cache()
        require_host_memory(WORLD * TOTAL * 4 * 5 // 4, f"decoder {kind}")
        g0 = _draw(0)
        torch.cuda.synchronize()
        want = host_snapshot(g0)
        if kind == "no_sync":
            for m in range(1, MICRO):
                gm = _draw(m)
                for r in range(WORLD):
                    row = host_snapshot(gm[r:r + 1])[0]
                    oracle.accumulate(want[r], row, oracle.F32)
                del gm
        grads = _views(want)
        if kind in ("sync", "no_sync"):
            b_of, off, bn = oracle.ddp_sync(grads, oracle.F32, MiB, 25 * MiB)
        elif kind == "bf16_hook":
            b_of, off, bn = oracle.ddp_sync_bf16_hook(grads, MiB, 25 * MiB)
        else:
            b_of, off, bn = oracle.ddp_sync_fp16_hook(grads, MiB, 25 * MiB)
        assert len(bn) == 37
        _case[kind] = (g0, want)
    return _case[kind]


def _plan():
    plan = ddp.ddp_plan_buckets(NUMELS, ddp.F32, MiB, 25 * MiB)
    assert len(plan[2]) == 37
    return plan


def _buckets(plan, dtype):
    """Every rank's bucket buffers, each between canary regions: (storages, buffers)."""
    storages, bk = [], []
    for _ in range(WORLD):
        row = []
        for n in plan[2]:
            st, b = guarded((int(n),), dtype)
            storages.append(st)
            row.append(b)
        bk.append(row)
    return storages, bk


def _run(kind, algo, via="sync_buckets"):
    g0, want = _expected(kind)
    g_storage, g = guarded_copy(g0)
    if kind == "no_sync":
        for m in range(1, MICRO):
            gm = _draw(m)
            ddp.ddp_grad_accumulate(g, gm)
            torch.cuda.synchronize()
            del gm
    plan = _plan()
    bk, bk_storages = None, []
    if algo in (ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_STAGED):
        bk_storages, bk = _buckets(plan, torch.float32)
    elif algo == ddp.DDP_ALGO_BF16_HOOK:
        bk_storages, bk = _buckets(plan, torch.bfloat16)
    views = _views(g)
    if via == "sync_buckets":
        ddp.ddp_sync_buckets(views, plan, bk, algo=algo)
    else:
        red = ddp.Reducer(views, plan, bk, algo=algo, comm_stream=torch.cuda.Stream())
        red.prepare()
        for p in range(len(NUMELS) - 1, -1, -1):       # backward makes the last-registered ready first
            red.mark_ready(p, torch.cuda.current_stream())
        red.finalize(torch.cuda.current_stream())
    torch.cuda.synchronize()
    if via != "sync_buckets":
        red.close()
    assert_canaries(g_storage, f"decoder gradients algo={algo}")
    for st in bk_storages:
        assert_canaries(st, f"decoder bucket algo={algo}")
    del bk, bk_storages
    assert_device_equals_host(g, want, f"decoder {kind} algo={algo} via {via}")
    assert ddp.ddp_device_status() == 0


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_VIEW, ddp.DDP_ALGO_STAGED])
def test_decoder_355m_n8_step_full(algo):
    _run("sync", algo)


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_VIEW])
def test_decoder_355m_n8_reducer_full(algo):
    _run("sync", algo, via="reducer")


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_BF16_HOOK, ddp.DDP_ALGO_BF16_HOOK_VIEW])
def test_decoder_355m_n8_bf16_hook_full(algo):
    _run("bf16_hook", algo)


def test_decoder_355m_n8_fp16_hook_view_full():
    _run("fp16_hook", ddp.DDP_ALGO_FP16_HOOK_VIEW)


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_VIEW])
def test_decoder_355m_n8_no_sync_full(algo):
    _run("no_sync", algo)
