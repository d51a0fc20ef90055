"""bench.py's replica path with two gloo ranks on the CPU: the barrier around
the timed region, the maximum of the ranks' times, the whole-job throughput
over all ranks' units and a single JSON line from rank 0.  Each rank's timed
region is a stand-in that sleeps and reports its own (different) duration,
so no GPU is involved; the functions under test are the ones bench.py's
timed steps and end-to-end leg run through."""
import contextlib
import io
import json
import os
import socket
import time

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    entered = []

    def run():
        # the other rank must have reached the barrier before this runs
        entered.append(time.time())
        time.sleep(0.05 * (rank + 1))
        return [12.5, 20.0][rank]

    ms = bench.timed_over_ranks(dist, torch.device("cpu"), run)
    value = bench.job_throughput(world, 1000.0, 4, ms)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.emit(rank, {"value": value, "ms": ms, "rank": rank})
    stamps = [None] * world
    dist.all_gather_object(stamps, entered[0])
    q.put((rank, ms, value, buf.getvalue(), stamps))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_time_and_one_line():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, ms, value, out, stamps = q.get(timeout=120)
        res[rank] = (ms, value, out, stamps)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest replica's time
    assert res[0][0] == res[1][0] == 20.0
    # whole-job throughput: 2 ranks x 1000 units x 4 steps in 20 ms
    assert res[0][1] == res[1][1] == 2 * 1000.0 * 4 / 20e-3
    # exactly one JSON line, from rank 0
    lines = [l for l in res[0][2].splitlines() if l.strip()]
    assert len(lines) == 1 and json.loads(lines[0])["rank"] == 0
    assert res[1][2] == ""
    # the barrier before the timed region: both entered within a moment
    a, b = res[0][3]
    assert abs(a - b) < 0.25
