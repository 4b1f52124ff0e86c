"""The multi-GPU path is replicas only (the layer chain is sequential and the pages' system is
single-GPU): N independent replicas, a barrier around the timed region and the max of the
per-rank times. This checks that host-side logic with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, dist = bench.dist_setup(world)
    dist.barrier()
    t = bench.max_over_ranks(dist, 10.0 + 5.0 * r)  # per-rank step time in ms
    q.put((r, w, t))
    dist.destroy_process_group()


def test_two_replicas_take_the_max_time():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in ps)
    out = sorted(q.get(timeout=10) for _ in range(2))
    assert out == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_process_needs_no_process_group():
    import bench

    saved = os.environ.pop("RANK", None)
    try:
        assert bench.dist_setup(1) == (0, 1, None)
        assert bench.max_over_ranks(None, 3.5) == 3.5
    finally:
        if saved is not None:
            os.environ["RANK"] = saved
