"""The bench's multi-GPU path on CPU ranks (gloo, world size 2): each rank
takes its own decoder layer (no data-path collective), and the reported
time is the maximum over ranks, so the whole-job value divides the bytes of
all ranks by the slowest rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank-dependent local timings: rank 0 slower on the first, rank 1 on the second
        got = bench.max_over_ranks([10.0 + rank, 7.0 - 3 * rank], torch.device("cpu"))
        q.put((rank, got, bench.rank_layer(rank)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_max_timing_and_take_distinct_layers():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [[11.0, 7.0], [11.0, 7.0]]
    assert {o[2] for o in out} == {0, 1}


def test_job_value_counts_every_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_value(1e9, 10, 20.0, 1)
    assert bench.job_value(1e9, 10, 20.0, 2) == pytest.approx(2 * one)
    assert one == pytest.approx(1e9 * 10 / 0.02 / 1e9)


def test_single_rank_max_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.25], torch.device("cpu")) == [3.5, 1.25]
