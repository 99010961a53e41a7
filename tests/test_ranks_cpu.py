"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The write path shards with no data exchange: each rank writes its own batch
into its own GPU's caches. Across ranks the benchmark only needs a barrier
around the timed region and the maximum elapsed time, which is what this
test exercises, together with the whole-job throughput arithmetic."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    d = bench.Dist()
    d.init("gloo")
    try:
        d.barrier()
        elapsed_ms = 10.0 + 5.0 * rank           # rank 1 is the slow one
        worst = d.max(elapsed_ms)
        tokens_per_rank, steps = 256, 100
        value = d.world * tokens_per_rank * steps / (worst / 1e3)
        out.put((rank, d.world, worst, value))
        d.barrier()
    finally:
        d.close()


def test_two_ranks_take_the_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, w, worst, value in res:
        assert w == 2 and worst == pytest.approx(15.0)
        assert value == pytest.approx(2 * 256 * 100 / 0.015)


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist()
    d.init("gloo")                 # no process group for one rank
    assert (d.world, d.rank, d.pg) == (1, 0, None)
    assert d.max(3.5) == 3.5


def test_bench_arguments():
    import bench
    a = bench.parse_args([])
    assert a.workload == "strided" and a.impl == "ours" and a.warmup >= 3 and a.suite == "all"
    a = bench.parse_args(["--impl", "reference", "--steps", "7", "--warmup", "4"])
    assert (a.steps, a.warmup) == (7, 4)
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
