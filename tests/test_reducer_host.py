"""The reducer's readiness bookkeeping, on the host (DDP_ALGO_DRYRUN: no CUDA).

Rules ("DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03
"Overlap"; "Day 17 · 梯度的集体行动" Reducer pseudo-code): a bucket is
launched once all its gradients are ready, buckets are launched in bucket
order (bucket i+1 never before bucket i), and the pass can only finish once
every bucket was launched.
"""
import numpy as np
import pytest

import gradient_sync_plan_gb300 as ddp
import workloads

MiB = 1 << 20


def _dry(numels, first=MiB, cap=25 * MiB):
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, first, cap)
    red = ddp.Reducer(None, plan, algo=ddp.DDP_ALGO_DRYRUN, world=2, numels=numels)
    return red, plan


def _expected_prefix(ready, n_buckets):
    k = 0
    while k < n_buckets and ready[k]:
        k += 1
    return list(range(k))


@pytest.mark.parametrize("seed", range(25))
def test_launch_order_is_bucket_order_and_as_early_as_possible(seed):
    rng = np.random.default_rng(seed)
    numels = [int(v) for v in rng.integers(1, 4000, size=int(rng.integers(1, 40)))]
    red, (b_of, off, bn) = _dry(numels, first=4000, cap=12000)
    K = len(bn)
    remaining = [int(np.sum(b_of == k)) for k in range(K)]
    ready = [False] * K
    for p in rng.permutation(len(numels)):
        red.mark_ready(int(p), stream=0)
        remaining[b_of[p]] -= 1
        if remaining[b_of[p]] == 0:
            ready[b_of[p]] = True
        assert red.launch_order() == _expected_prefix(ready, K)
    red.finalize(stream=0)
    assert red.launch_order() == list(range(K))


def test_reverse_registration_order_launches_each_bucket_at_its_last_gradient():
    numels = workloads.param_numels(workloads.decoder_param_shapes())
    red, (b_of, off, bn) = _dry(numels)
    launched_at = {}
    for p in range(len(numels) - 1, -1, -1):          # backward order
        before = len(red.launch_order())
        red.mark_ready(p, stream=0)
        after = red.launch_order()
        for k in after[before:]:
            launched_at[k] = p
    red.finalize(stream=0)
    assert red.launch_order() == list(range(len(bn)))
    # bucket k is launched exactly when its lowest-index (last in backward) member is ready
    for k in range(len(bn)):
        assert launched_at[k] == int(np.min(np.nonzero(b_of == k)[0]))


def test_double_mark_and_missing_gradient_are_errors():
    numels = [100, 200, 300]
    red, (b_of, off, bn) = _dry(numels, first=400, cap=400)
    red.mark_ready(2, stream=0)
    with pytest.raises(ddp.DDPError):
        red.mark_ready(2, stream=0)
    red.mark_ready(1, stream=0)
    with pytest.raises(ddp.DDPError):                 # parameter 0 never got a gradient
        red.finalize(stream=0)
    red.prepare()                                      # a new pass starts clean
    for p in (2, 1, 0):
        red.mark_ready(p, stream=0)
    red.finalize(stream=0)
    assert red.launch_order() == list(range(len(bn)))
    with pytest.raises(ddp.DDPError):
        red.mark_ready(7, stream=0)
    red.close()


def test_inconsistent_plans_are_refused_when_the_reducer_is_created():
    numels = [100, 200, 300]
    b_of, off, bn = ddp.ddp_plan_buckets(numels, ddp.F32, 400, 400)
    bad_plans = [
        (b_of, [o + 1 if i == 0 else o for i, o in enumerate(off)], bn),        # a member runs past its bucket
        (b_of, off, [n - 1 for n in bn]),                                          # bucket too short
        ([0, 0, 0], [0, 50, 0], [600]),                                            # two members overlap
        (b_of, [-1] + list(off[1:]), bn),                                          # negative offset
    ]
    for plan in bad_plans:
        with pytest.raises(ddp.DDPError):
            ddp.Reducer(None, plan, algo=ddp.DDP_ALGO_DRYRUN, world=2, numels=numels)


def test_bucket_times_in_a_dry_run_are_unmeasured():
    numels = [100, 200, 300]
    red, (b_of, off, bn) = _dry(numels, first=400, cap=400)
    for p in (2, 1, 0):
        red.mark_ready(p, stream=0)
    red.finalize(stream=0)
    assert red.bucket_times() == [-1.0] * len(bn)
    red.close()


def test_reducer_cta_budget_validates():
    # -1 follows the process-wide cap, 0 removes any cap, n > 0 caps; below -1
    # and a NULL reducer are refused (host only: a dry-run reducer)
    red, _ = _dry([10, 20, 30])
    for ok in (-1, 0, 1, 38, 1 << 20):
        red.set_max_ctas(ok)
    with pytest.raises(ddp.DDPError):
        red.set_max_ctas(-2)
    assert ddp.lib().ddp_reducer_set_max_ctas(None, 4) == -1
    red.prepare()
    for p in range(2, -1, -1):
        red.mark_ready(p, stream=0)
    red.finalize(stream=0)
    red.close()
