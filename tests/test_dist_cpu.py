"""The N > 1 host logic of bench.py, on CPU with the gloo backend (world size 2).

bench.py under torchrun runs one independent replica per rank (the path shards by
sequence with no data-path collective); the only cross-rank operations are the
barriers around the timed region and the max over ranks of the step time, from which
rank 0 computes the whole-job throughput.  These run here as two spawned processes.
The reference arm's non-zero ranks exit without work.
"""
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w = bench.dist_init("gloo")
    bench.barrier()
    local_ms = 1.5 if rank == 0 else 4.25          # the slower rank decides the time
    ms = bench.max_over_ranks(local_ms)
    bench.barrier()
    a = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    rc = bench.run_reference(a) if rank != 0 else None   # rank != 0: exits without work
    q.put((r, w, ms, rc))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_timing_max_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == pytest.approx(4.25) for r in res)
    assert res[1][3] == 0


def test_single_process_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    bench.barrier()
    assert bench.dist_env()[1] >= 1
