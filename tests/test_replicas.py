"""Multi-process host logic of the replica path on CPU (gloo, world_size 2)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from mla_position_independent_gb300 import replicas, synth


def test_request_shard_partitions():
    for B in (1, 7, 8, 64):
        for world in (1, 2, 3, 8):
            got = [replicas.request_shard(B, r, world) for r in range(world)]
            assert got[0][0] == 0 and got[-1][1] == B
            assert all(got[i][1] == got[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in got]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = synth.custom_case([[(0, 32, 0, 0), (100, 40 + 8 * b, 7, 1)] for b in range(5)],
                             n_rows=400, n_q=0)
    lo, hi = replicas.request_shard(case.B, rank, world)
    sub, ip = replicas.subtable(case.chunks, case.indptr, lo, hi)
    from mla_position_independent_gb300 import build
    build.build()
    import mla_position_independent_gb300 as irm
    ctx = irm.validate_chunks(sub, ip, 400)      # each shard is a valid table on its own
    t = replicas.max_over_ranks(10.0 + rank, world)
    ids = torch.zeros(case.B, dtype=torch.int64)
    ids[lo:hi] = 1
    dist.all_reduce(ids)
    q.put((rank, list(ctx), t, ids.tolist()))
    dist.destroy_process_group()


def test_replicas_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, ctx0, t0, ids0), (_, ctx1, t1, ids1) = res
    assert t0 == t1 == 11.0                      # the slowest rank's time
    assert ids0 == ids1 == [1] * 5               # every request on exactly one rank
    assert ctx0 + ctx1 == [72 + 8 * b for b in range(5)]
