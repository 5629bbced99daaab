"""The benchmark's multi-rank path on CPU: two gloo ranks, each a replica,
agree on the max-over-ranks time and the barrier; rank 0 alone would print.
(The data path has no collective: replicas share nothing but timing.)"""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + rank * 2.5, w)
    # weak scaling: every rank did one unit of work in at most t
    value = w * 1.0 / t
    dist.destroy_process_group()
    q.put((r, w, t, value))


def test_two_rank_timing_reduction():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[2] == pytest.approx(3.5) for r in res)     # max over ranks, seen by both
    assert all(r[3] == pytest.approx(2 / 3.5) for r in res)


def test_reference_arm_sample_is_bounded():
    """The oracle sample the CPU baseline times is one expert of the MoE
    workload and reports a positive rate with its core count."""
    import bench
    v, desc, cores = bench.oracle_sample(seconds_hint=0.0)
    assert v > 0 and cores >= 1 and "2048 rows" in desc
    v, desc, cores = bench.oracle_sample(seconds_hint=0.0, rows=512)
    assert "512 rows" in desc


def test_clock_summary_uses_the_timed_window():
    """Clock samples are time-stamped: the summary takes those inside the
    timed region, and falls back to all samples (flagged) when the region
    was shorter than the sampling interval."""
    import bench
    c = bench.ClockSampler(0)
    c.lines = [(1.0, "0, 2000, 2070, 500, Not Active, Not Active, Not Active, Active"),
               (5.0, "0, 1900, 2070, 900, Not Active, Not Active, Not Active, Not Active"),
               (5.5, "0, 1950, 2070, 950, Not Active, Not Active, Not Active, Not Active")]
    c.t_start, c.t_end = 4.0, 6.0
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1925.0 and s["reasons"] == [] and s["window"] == "timed region"
    c.t_start, c.t_end = 7.0, 8.0
    s = c.summary()
    assert s["samples"] == 3 and "sw_power_cap" in s["reasons"] and s["window"].startswith("around")
