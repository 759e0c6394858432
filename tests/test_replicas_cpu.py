"""The multi-process path of bench.py on CPU: world-size-2 gloo ranks.

The scan does not shard without a collective in the backward (dB / dC sum
over every channel, dA / dD / ddelta_bias over every batch), so multi-GPU
runs are independent replicas.  The process group only carries the barrier
and the max-over-ranks timing; these ranks check that coordination and the
whole-job throughput formula, and that the reference arm does no work on
ranks other than 0.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    try:
        w, r, local = bench.dist_setup("gloo")
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(w)
        local_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, w, device="cpu")
        value = bench.job_throughput(1000, w, ms)
        dist.destroy_process_group()
        q.put((rank, ms, value))
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, "error", repr(e)))


@pytest.mark.timeout(120)
def test_two_gloo_replicas_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 20.0, (rank, ms, value)  # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 1000 / 0.020)  # both replicas' units over that time


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 1, 3

    bench.run_reference(Args())  # returns at once: no oracle work, no output
    assert capsys.readouterr().out == ""
