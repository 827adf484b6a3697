"""The multi-rank bench logic on CPU: two gloo ranks, max-over-ranks timing,
per-rank workloads (own seed, same shapes) and the whole-job aggregate."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        m = bench.dist_max(ms)
        w = bench.rank_workload(bench.synth.T1024, rank)
        q.put((rank, m, w.seed, w.T, bench.aggregate_tokens_per_s(w, world, m)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_aggregate():
    import multiprocessing as mp

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
    (r0, m0, s0, T0, v0), (r1, m1, s1, T1, v1) = res
    assert m0 == m1 == 15.0
    assert s0 != s1 and T0 == T1
    assert v0 == v1 == pytest.approx(2 * T0 / 15e-3)


def test_single_process_is_identity():
    import bench

    assert bench.dist_max(3.5) == 3.5
