"""GPU parity of the overlapped reducer (ddp_reducer_*) against the oracle.

A synthetic backward writes each parameter's gradient (all ranks) on a
compute stream, in reverse registration order or in a shuffled order, and
marks it ready; the reducer syncs buckets on a separate comm stream as they
complete.  After finalize, every gradient must equal the oracle's DDP step
(plan -> pack -> ring allreduce / N -> unpack) bit for bit.
"""
import numpy as np
import pytest
import torch

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads
from gpu_util import assert_bits_equal, f32_or_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_VIEW, ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_STAGED])
@pytest.mark.parametrize("order", ["backward", "shuffled"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_overlapped_reducer_matches_oracle(algo, order, dtype):
    numels = workloads.param_numels(workloads.decoder_param_shapes(n_layer=4, d_model=128, d_ff=512, vocab=2000,
                                                                   n_pos=128))
    world, first, cap = 8, 64 << 10, 256 << 10
    code = ddp.BF16 if dtype == "bf16" else ddp.F32
    plan = ddp.ddp_plan_buckets(numels, code, first, cap)
    assert len(plan[2]) > 5
    src = workloads.rank_vectors(world, sum(numels), "randn", std=1e-2, dtype=dtype, seed0=3)
    src_h = f32_or_bits(src)
    offs = np.cumsum([0] + numels)
    grads_h = [[src_h[r, offs[p]:offs[p + 1]].copy() for p in range(len(numels))] for r in range(world)]
    oracle.ddp_sync(grads_h, code, first, cap)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])

    src_d = src.cuda()
    g = torch.zeros_like(src_d)
    views = [[g[r, int(offs[p]):int(offs[p + 1])] for p in range(len(numels))] for r in range(world)]
    buckets = None
    if algo != ddp.DDP_ALGO_VIEW:
        buckets = [[torch.empty(int(n), dtype=src_d.dtype, device="cuda") for n in plan[2]] for _ in range(world)]
    comm, compute = torch.cuda.Stream(), torch.cuda.Stream()
    red = ddp.Reducer(views, plan, buckets, algo=algo, comm_stream=comm)
    torch.cuda.synchronize()
    for _ in range(2):                                    # two passes: prepare() resets readiness
        g.zero_()
        torch.cuda.synchronize()
        red.prepare()
        params = list(range(len(numels) - 1, -1, -1))
        if order == "shuffled":
            params = list(np.random.default_rng(5).permutation(len(numels)))
        with torch.cuda.stream(compute):
            for p in params:
                a, b = int(offs[p]), int(offs[p + 1])
                g[:, a:b].copy_(src_d[:, a:b])            # "backward" produces grad p on every rank
                red.mark_ready(int(p), compute)
        red.finalize(torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert red.launch_order() == list(range(len(plan[2])))
        assert_bits_equal(f32_or_bits(g), want, f"reducer algo={algo} order={order}")
        times = red.bucket_times()                        # per-bucket sync time on the comm stream
        assert len(times) == len(plan[2]) and all(t > 0 for t in times), times
    red.close()


def test_bucket_times_are_unmeasured_inside_a_captured_graph():
    # timing events cannot be recorded while the comm stream is captured: a
    # pass captured into a graph reports -1 per bucket, a plain pass real times
    numels = workloads.param_numels(workloads.decoder_param_shapes(n_layer=2, d_model=64, d_ff=256, vocab=500,
                                                                   n_pos=32))
    world = 4
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, 4096, 40000)
    g = workloads.rank_vectors(world, sum(numels), "randn", std=1e-2, seed0=8).cuda()
    offs = np.cumsum([0] + numels)
    views = [[g[r, int(offs[p]):int(offs[p + 1])] for p in range(len(numels))] for r in range(world)]
    comm, compute = torch.cuda.Stream(), torch.cuda.Stream()
    red = ddp.Reducer(views, plan, None, algo=ddp.DDP_ALGO_VIEW, comm_stream=comm)

    def one_pass():
        red.prepare()
        for p in range(len(numels) - 1, -1, -1):
            red.mark_ready(p, compute)
        red.finalize(compute)

    one_pass()
    torch.cuda.synchronize()
    assert all(t > 0 for t in red.bucket_times())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=compute):
        one_pass()
    assert red.bucket_times() == [-1.0] * len(plan[2])
    graph.replay()
    torch.cuda.synchronize()
    red.close()


@pytest.mark.parametrize("algo", [ddp.DDP_ALGO_VIEW, ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_BF16_HOOK_VIEW])
def test_reducer_with_its_own_cta_budget_matches_oracle(algo):
    # a reducer capped at 19 CTAs (while the process-wide cap stays unset)
    # gives the oracle's bits, and leaves other calls uncapped: the budget is
    # this reducer's own
    numels = workloads.param_numels(workloads.decoder_param_shapes(n_layer=4, d_model=128, d_ff=512, vocab=2000,
                                                                   n_pos=128))
    world, first, cap = 8, 64 << 10, 1 << 20
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, first, cap)
    src = workloads.rank_vectors(world, sum(numels), "randn", std=1e-2, seed0=17)
    src_h = f32_or_bits(src)
    offs = np.cumsum([0] + numels)
    grads_h = [[src_h[r, offs[p]:offs[p + 1]].copy() for p in range(len(numels))] for r in range(world)]
    if algo == ddp.DDP_ALGO_BF16_HOOK_VIEW:
        oracle.ddp_sync_bf16_hook(grads_h, first, cap)
    else:
        oracle.ddp_sync(grads_h, oracle.F32, first, cap)
    want = np.stack([np.concatenate(grads_h[r]) for r in range(world)])
    g = src.cuda()
    views = [[g[r, int(offs[p]):int(offs[p + 1])] for p in range(len(numels))] for r in range(world)]
    buckets = None
    if algo == ddp.DDP_ALGO_FUSED:
        buckets = [[torch.empty(int(n), device="cuda") for n in plan[2]] for _ in range(world)]
    assert ddp.ddp_set_max_ctas(0) == 0
    red = ddp.Reducer(views, plan, buckets, algo=algo, comm_stream=torch.cuda.Stream())
    red.set_max_ctas(19)
    red.prepare()
    compute = torch.cuda.current_stream()
    for p in range(len(numels) - 1, -1, -1):
        red.mark_ready(p, compute)
    red.finalize(compute)
    torch.cuda.synchronize()
    red.close()
    assert_bits_equal(f32_or_bits(g), want, f"reducer with 19 CTAs algo={algo}")
    assert ddp.ddp_set_max_ctas(0) == 0                 # the process-wide cap was never touched
    with pytest.raises(ddp.DDPError):
        red2 = ddp.Reducer(views, plan, buckets, algo=algo, comm_stream=torch.cuda.Stream())
        try:
            red2.set_max_ctas(-2)
        finally:
            red2.close()
