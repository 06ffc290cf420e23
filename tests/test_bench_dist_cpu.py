"""Host logic of bench.py's multi-process path (replicas only), run as two
gloo ranks on the CPU: barrier, max over ranks, whole-job aggregation."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist()
    d.barrier()
    elapsed = [0.5, 2.0][rank]          # rank 1 is the slow one
    el_max = d.max(elapsed)
    value = bench.aggregate(1000.0, el_max, d.world)
    q.put((rank, el_max, value))
    d.close()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, el_max, value in out:
        assert el_max == 2.0                 # max over ranks
        assert value == pytest.approx(1000.0 * 2 / 2.0)   # all ranks' units / slowest time


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.rank == 0 and d.max(3.0) == 3.0
    assert bench.aggregate(10.0, 2.0, 1) == 5.0
    args = bench.parse_args([])
    assert args.steps >= 1 and args.warmup >= 3 and args.impl == "ours"
