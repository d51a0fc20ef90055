"""Row sharding over two ranks (gloo, CPU): every rank computes its segments
of ln_modulate / rmsnorm_silu_cl with the oracle, rank 0 gathers them, and
the result must equal the single-process result bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from rmsnorm_modulate_gb300.sharding import row_range, row_segments


def test_row_range_partition():
    for rows in (0, 1, 7, 100, 4608):
        for world in (1, 2, 3, 8):
            ranges = [row_range(rows, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == rows
            for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_row_segments_cut_at_batch_boundaries():
    B, S = 3, 10
    for world in (1, 2, 4, 7):
        seen = []
        for r in range(world):
            for b, s0, s1 in row_segments(B, S, r, world):
                assert 0 <= s0 < s1 <= S and 0 <= b < B
                seen.extend(b * S + s for s in range(s0, s1))
        assert seen == list(range(B * S))


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
    import oracle
    import workloads as W

    inp = W.ln_modulate_inputs(2, 37, 256, seed=1, per_batch_mod=True)
    parts = []
    for b, s0, s1 in row_segments(2, 37, rank, world):
        out, mean, rstd = oracle.ln_modulate(np.ascontiguousarray(inp["x"][b:b + 1, s0:s1]),
                                             inp["scale"][b], inp["shift"][b])
        parts.append((b, s0, s1, out, mean, rstd))
    gathered = [None] * world
    dist.all_gather_object(gathered, parts)
    if rank == 0:
        full, fmean, frstd = oracle.ln_modulate(inp["x"], inp["scale"], inp["shift"])
        got = np.empty_like(full)
        gmean = np.empty_like(fmean)
        grstd = np.empty_like(frstd)
        for rp in gathered:
            for b, s0, s1, out, mean, rstd in rp:
                got[b, s0:s1] = out[0]
                gmean[b * 37 + s0:b * 37 + s1] = mean
                grstd[b * 37 + s0:b * 37 + s1] = rstd
        q.put(bool(np.array_equal(got, full) and np.array_equal(gmean, fmean)
                   and np.array_equal(grstd, frstd)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sharded_result_equals_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok
