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


def test_reference_arm_json_contract(monkeypatch):
    """The reference arm (the oracle on the host cores) prints the same line
    as ours, marked impl=reference, with its own CPU baseline and zero e2e copies."""
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = bench.run_reference(args, bench.Dist())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["warmup"] >= 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
