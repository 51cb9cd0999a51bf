"""Multi-process (world size 2, gloo, CPU) check of bench.py's replica plumbing.

The method shards by independent requests, heads and row blocks, so a multi-GPU run is N
independent replicas with no collective on the data path; the only cross-rank steps are
the barriers around the timed region and the reductions of the reported numbers (time:
max over ranks; bytes: sum over ranks). This runs those helpers in two processes.
"""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    try:
        import bench
        dist, r, w = bench.dist_setup(ws)
        bench.barrier(dist)
        t_max = bench.max_over_ranks(dist, 1.5 + r)          # per-rank "times"
        total = bench.sum_over_ranks(dist, 100.0 * (r + 1))  # per-rank "bytes"
        bench.barrier(dist)
        q.put((r, w, t_max, total))
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001 - report to the parent
        q.put(("error", repr(e)))


def test_replica_reductions_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    assert all(r[0] != "error" for r in res), res
    got = sorted(res)
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    # every rank sees the max time and the summed bytes
    assert all(g[2] == pytest.approx(2.5) for g in got)
    assert all(g[3] == pytest.approx(300.0) for g in got)
    # value = bytes of all ranks / max-over-ranks time
    assert got[0][3] / got[0][2] == pytest.approx(120.0)


def test_single_process_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    dist, r, w = bench.dist_setup(1)
    assert dist is None and r == 0 and w == 1
    assert bench.max_over_ranks(None, 3.0) == 3.0 and bench.sum_over_ranks(None, 4.0) == 4.0
