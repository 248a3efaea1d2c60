"""Failure detection among host processes (gloo on the CPU, no GPU).

A ring hangs without an error when its ranks disagree: one rank that never
joins a step, or ranks whose bucket plans differ and so issue different
collective sequences ("Day 17 · 梯度的集体行动", the question on why DDP can
hang without reporting anything).  These tests make both failures on the
host, one process per rank, and check that every surviving rank stops with
an error instead of waiting forever:

  * plan mismatch: ranks exchange ddp_plan_fingerprint before the first
    sync; one rank registered an extra parameter, so every rank sees the
    mismatch and stops;
  * a rank that never joins: it exits before the step; the other ranks'
    collective fails (peer closed, or the short process-group timeout) and
    they stop.

Each worker writes its outcome to a file; the test reads them after the
processes have ended.
"""
import datetime
import os
import socket
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import gradient_sync_plan_gb300 as ddp
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=timeout_s))


def _plan_worker(rank, world, port, odd_rank, out_dir):
    _init(rank, world, port, 30)
    outcome = "unknown"
    try:
        numels = workloads.param_numels(workloads.decoder_param_shapes(n_layer=2, d_model=64, d_ff=256,
                                                                       vocab=500, n_pos=32))
        if rank == odd_rank:
            numels = numels + [64]                 # this rank registered one more parameter
        plan = ddp.ddp_plan_buckets(numels, ddp.F32, 4096, 40000)
        fp = ddp.ddp_plan_fingerprint(numels, plan, ddp.F32)
        mine = torch.tensor([fp & 0x7FFFFFFFFFFFFFFF, fp >> 63], dtype=torch.int64)
        gathered = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(gathered, mine)
        same = all(torch.equal(g, gathered[0]) for g in gathered)
        outcome = "consistent" if same else "mismatch"
    except Exception as e:                         # noqa: BLE001 -- the outcome is what the test checks
        outcome = "error: " + type(e).__name__
    finally:
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(outcome)
        dist.destroy_process_group()


@pytest.mark.parametrize("odd_rank", [None, 2])
def test_plan_fingerprints_expose_a_rank_with_a_different_plan(tmp_path, odd_rank):
    world = 3
    mp.start_processes(_plan_worker, args=(world, _free_port(), odd_rank, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    outcomes = [(tmp_path / f"r{r}.txt").read_text() for r in range(world)]
    want = "consistent" if odd_rank is None else "mismatch"
    assert outcomes == [want] * world, outcomes


def _absent_worker(rank, world, port, out_dir):
    _init(rank, world, port, 5)
    if rank == world - 1:
        # this rank leaves before the step, between collectives, and never joins
        os._exit(0)
    outcome = "unknown"
    try:
        x = torch.ones(1024)
        dist.all_reduce(x)
        outcome = "completed"
    except Exception as e:                         # noqa: BLE001
        outcome = "error: " + type(e).__name__
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(outcome)
    os._exit(0)


def test_a_rank_that_never_joins_is_detected_not_waited_for(tmp_path):
    world = 3
    ctx = mp.start_processes(_absent_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                             start_method="spawn", join=False)
    deadline = time.monotonic() + 120
    done = False
    try:
        while not done and time.monotonic() < deadline:
            done = ctx.join(timeout=max(1.0, deadline - time.monotonic()))
    finally:
        for p in ctx.processes:          # never leave a waiting rank behind
            if p.is_alive():
                p.terminate()
    assert done, "a surviving rank was still waiting after 120 s"
    for r in range(world - 1):
        out = (tmp_path / f"r{r}.txt").read_text()
        assert out.startswith("error"), (r, out)
