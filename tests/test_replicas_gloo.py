"""The N>1 bench path runs independent replicas (no collective on the data
path): ranks meet at barriers and the timing is the max over ranks.  Checked
here with two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    bench.barrier(ws)
    per_call_ms = 1.0 + rank            # rank 1 is the slow replica
    worst = bench.allmax(per_call_ms, ws)
    whole_job_us = worst * 1000.0 / ws  # ws calls complete in parallel
    bench.barrier(ws)
    dist.destroy_process_group()
    q.put((rank, worst, whole_job_us))


@pytest.mark.timeout(120)
def test_two_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(30)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]        # both ranks see the max
    assert res[0][2] == pytest.approx(1000.0)
