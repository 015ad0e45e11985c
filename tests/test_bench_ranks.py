"""The benchmark's N>1 path on CPU: two gloo ranks agree on the slowest rank's time and
on the whole-job throughput (replicas of independent work, no data exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    my_time = 1.0 + rank            # rank 1 is the slower one
    bench.barrier(dist)
    t = bench.max_over_ranks(dist, my_time)
    value = bench.combine(100.0, w, t)
    q.put((r, w, t, value))
    dist.destroy_process_group()


def test_two_gloo_ranks():
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
    assert [r[0] for r in res] == [0, 1]
    for r, w, t, value in res:
        assert w == 2 and t == 2.0 and value == pytest.approx(100.0)


def test_single_rank_defaults(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.combine(10.0, 1, 2.0) == 5.0
    args = bench.parse_args([])
    assert args.gpus == 1 and args.warmup >= 3
