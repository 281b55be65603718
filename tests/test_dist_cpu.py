"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timed
region's max over ranks, and the reference arm printing on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + 5 * rank)
    ws, r, local = bench.dist_env()
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, got, ws, r, local))


def test_max_over_ranks_gloo():
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
    assert [x[1] for x in res] == [15.0, 15.0]
    assert [(x[2], x[3], x[4]) for x in res] == [(2, 0, 0), (2, 1, 1)]


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_silent_on_other_ranks(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from exact_attention_57_gb300.workloads import WORKLOADS
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 3
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A(), WORKLOADS["b1h1n256d64-f32-simt"])
    assert buf.getvalue() == ""
