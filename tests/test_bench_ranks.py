"""Multi-rank logic of bench.py on CPU: world_size-2 gloo ranks (no GPU).

Under torchrun every rank runs an independent replica of the layer; the job
time is the slowest rank's, and the throughput counts every rank's tokens.
The reference arm runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r measured (1 + r) ms per step and (10 - r) ms end to end
        ms, e2e = bench.max_over_ranks([1.0 + rank, 10.0 - rank], world)
        value = bench.job_tokens_per_s(world, 1000, ms)

        class A:  # the reference arm's arguments; rank 1 must return without work
            workload, M, steps, warmup, ref_tokens = "tiny-int4", 16, 1, 1, 2
        ref = bench.run_reference(A, rank) if rank == 1 else "skipped"
        dist.barrier()
        q.put((rank, ms, e2e, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got = {r: (ms, e2e, v, ref) for r, ms, e2e, v, ref in out}
    for r in (0, 1):
        ms, e2e, v, _ = got[r]
        assert ms == 2.0 and e2e == 10.0           # max over ranks, seen by every rank
        assert v == pytest.approx(2 * 1000 / 2e-3)  # both ranks' tokens over the slowest time
    assert got[1][3] is None                        # reference arm: rank 1 does no work


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_tokens_per_s(1, 2304, 0.0657) == pytest.approx(2304 / 0.0657e-3)
