"""Host side of the multi-GPU mode (independent replicas, no data-path
collective), run as two gloo ranks on the CPU: the rank/world environment is
read as torchrun sets it, the job time is the maximum over ranks, and only
rank 0 runs and prints the reference (oracle) arm."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_info()
        bench.barrier(w)
        t = bench.max_over_ranks(1.5 + r, w)          # each replica's own time
        ref = None
        if r != 0:                                    # non-zero ranks do no reference work
            class A:
                steps, warmup = 1, 0
            ref = bench.run_reference(A())
        q.put((r, w, local, t, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_share_max_time_and_rank0_reports():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[:3] for o in out] == [(0, 2, 0), (1, 2, 1)]
    assert all(o[3] == 2.5 for o in out)              # the slowest replica's time
    assert out[1][4] is None                          # rank 1 ran no reference work
