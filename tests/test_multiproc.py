"""The multi-rank bench path on CPU: two gloo ranks (world size 2) run the
rank helpers bench.py uses under torchrun.  Each rank processes its own
replica of the workload (weak scaling, no data-path collective); the job
throughput is every rank's tokens over the slowest rank's time."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        import torch

        import bench
        r, n = bench.init_dist("gloo")
        assert (r, n) == (rank, ws)
        elapsed = [40.0, 55.0][rank]  # rank 1 is the slower one
        slowest = bench.max_over_ranks(elapsed)
        value = bench.aggregate(tokens_per_rank_step=1000, steps=5, elapsed_ms_max=slowest, n_ranks=n)
        bench.barrier()
        torch.distributed.destroy_process_group()
        q.put((rank, slowest, value))
    except Exception as e:  # noqa: BLE001
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    pytest.importorskip("torch.distributed")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest != "error", value
        assert slowest == 55.0  # every rank sees the max over ranks
        assert value == pytest.approx(2 * 5 * 1000 / 0.055)


def test_single_rank_helpers_are_identities():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate(10, 2, 1000.0, 1) == pytest.approx(20.0)
