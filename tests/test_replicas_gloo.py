"""The N>1 path of bench.py (independent replicas, host-side barrier and max-over-ranks
timing) on two CPU ranks over gloo.  No GPU."""
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
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each replica reports its own step time; the job time is the slowest rank's
    t = bench.max_over_ranks(10.0 + rank, w)
    q.put((rank, t))
    dist.destroy_process_group()


def test_two_rank_replicas_take_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_reference_arm_line(monkeypatch, capsys):
    """--impl reference prints one JSON line with the oracle as the baseline (tiny workload)."""
    import json
    import sys
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                                      "--workload", "tiny_256"])
    bench.main()
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
