"""The N > 1 path of the benchmark on CPU: world-size-2 gloo process groups.

Requests are independent, so N GPUs run N replicas with no collective on the
data path; the only cross-rank steps are the timing reductions of the
benchmark (slowest rank's time, units summed over ranks) and the reference
arm's "rank 0 alone runs" rule.  Both are host logic and run here on gloo.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms_per_rank, units_per_rank, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        rate, ms, total = bench.job_rate(ms_per_rank[rank], units_per_rank[rank], dist, "cpu")
        # the reference arm: every rank but 0 leaves at once without work
        skipped = bench.reference_arm(None, None, rank, world) is None if rank else None
        out_q.put((rank, rate, ms, total, skipped))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world, ms_per_rank, units_per_rank):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, ms_per_rank, units_per_rank, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_replicas_rate_uses_slowest_rank_and_all_units():
    ms = [250.0, 400.0]            # rank 1 is the slow replica
    units = [3000, 3000]           # weak scaling: same work per rank
    res = _run(2, ms, units)
    for rank, rate, ms_max, total, _ in res:
        assert ms_max == 400.0
        assert total == 6000
        assert rate == pytest.approx(6000 / 0.4)
    assert res[1][4] is True       # rank 1 did no reference work


def test_two_replicas_uneven_units():
    res = _run(2, [100.0, 100.0], [10, 30])
    for _, rate, ms_max, total, _ in res:
        assert total == 40 and ms_max == 100.0
        assert rate == pytest.approx(400.0)


def test_single_process_needs_no_group():
    import bench
    rate, ms, total = bench.job_rate(500.0, 1000)
    assert (rate, ms, total) == (2000.0, 500.0, 1000)
