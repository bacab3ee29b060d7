"""The N > 1 host path of bench.py, on CPU with two gloo ranks.

The data path has no collective: every rank runs the fused operators on its own shard (batch) of
the workload.  What crosses ranks is the barrier around the timed region and the maximum of the
ranks' times, from which the whole-job throughput is formed.  These tests run those pieces as two
processes (spawned, gloo backend, 127.0.0.1) and check them against what each rank computes alone.
"""
import os
import socket

import numpy as np
import pytest

import bench
import fc_inputs
import oracle

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # a per-rank time: the job's is the slowest rank's
        t = bench.max_over_ranks(torch, 1.5 + rank, dist, "cpu")
        # this rank's shard of a tiny conv -> GELU -> pool workload, computed by the oracle
        d = fc_inputs.conv_inputs(1, 2, 6, 7, 4, seeds=bench.rank_seeds(rank))
        y = oracle.conv3x3_act_pool(d["x"], d["w"], d["b"], "gelu")
        got = [torch.zeros(1, 4, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(got, torch.from_numpy(np.ascontiguousarray(y)))   # test-side comparison only
        dist.barrier()
        q.put((rank, t, [g.numpy() for g in got]))
    finally:
        dist.destroy_process_group()


def _run(world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda o: o[0])


def test_two_gloo_ranks_time_and_shards():
    out = _run(WORLD)
    # every rank sees the same job time: the maximum over ranks
    assert [o[1] for o in out] == [1.5 + WORLD - 1] * WORLD
    # the shards are distinct (own x seeds) and each is what that rank computes alone
    for rank in range(WORLD):
        d = fc_inputs.conv_inputs(1, 2, 6, 7, 4, seeds=bench.rank_seeds(rank))
        alone = oracle.conv3x3_act_pool(d["x"], d["w"], d["b"], "gelu")
        for o in out:
            np.testing.assert_array_equal(o[2][rank], alone)
    assert not np.array_equal(out[0][2][0], out[0][2][1])


def test_rank_seeds_share_weights_and_split_inputs():
    s0, s1 = bench.rank_seeds(0), bench.rank_seeds(1)
    assert s0[0] != s1[0] and s0[1:] == s1[1:]
    assert s0 == (fc_inputs.SEED_X, fc_inputs.SEED_W, fc_inputs.SEED_B)


def test_job_throughput_counts_every_rank_over_the_slowest_time():
    f = 7.6e10
    assert bench.job_tflops(f, 1, 0.5) == pytest.approx(f / 0.5e-3 / 1e12)
    assert bench.job_tflops(f, 4, 0.5) == pytest.approx(4 * bench.job_tflops(f, 1, 0.5))


def test_max_over_ranks_without_a_process_group_is_the_local_value():
    import torch
    assert bench.max_over_ranks(torch, 3.25, None, "cpu") == 3.25


def _lost_rank_main(rank, world, port, q):
    import datetime
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=4))
    if rank == 1:
        # this rank never joins the timed region's collective (a failure made on the host): it
        # idles past the group's timeout and leaves
        import time
        time.sleep(10)
        q.put((rank, "left"))
        return
    try:
        bench.max_over_ranks(torch, 1.0, dist, "cpu")
        q.put((rank, "completed"))
    except Exception as e:   # the waiting rank gets an error within the timeout, not a hang
        q.put((rank, f"error: {type(e).__name__}"))


def test_a_rank_that_leaves_is_reported_not_waited_for():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_lost_rank_main, args=(r, WORLD, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(WORLD))
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    assert out[1] == "left"
    assert out[0].startswith("error")
