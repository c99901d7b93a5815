"""bench.py's multi-rank plumbing on two CPU ranks over gloo (no GPU): the
barrier, the maximum of the ranks' timings that every rank then reports, and
the reference arm, which runs on rank 0 only (the other ranks return without
work)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, _ = bench.dist_env()
    dist = bench.dist_init(w, backend="gloo")
    bench.barrier(dist)
    ms = bench.max_over_ranks(dist, 10.0 + 3.0 * r)
    args = type("Args", (), {"steps": 1, "warmup": 3})()
    ref = bench.run_reference(args, r, w) if r != 0 else "rank 0"
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((r, w, ms, ref))


def test_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(i, 2, port, q)) for i in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[:2] for r in res] == [(0, 2), (1, 2)]
    assert [r[2] for r in res] == [13.0, 13.0]      # every rank reports the slowest rank's time
    assert res[1][3] is None                        # the reference arm does no work off rank 0


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.dist_init(1) is None
    assert bench.max_over_ranks(None, 4.5) == 4.5
    bench.barrier(None)
