"""Multi-rank host logic on CPU: world-size-2 gloo process group."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from linear_attention_speculative_gb300.replicas import max_over_ranks, shard


def test_shard_covers_every_sequence_once():
    for n in (0, 1, 5, 256, 257):
        for world in (1, 2, 3, 8):
            ranges = [shard(n, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c and b >= a
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = shard(257, rank, world)
    t = max_over_ranks(1.5 + rank)   # rank r "took" 1.5 + r ms
    n = max_over_ranks(float(hi - lo))
    out.put((rank, lo, hi, t, n))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_split():
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
    assert [(r[1], r[2]) for r in res] == [(0, 129), (129, 257)]
    assert all(r[3] == 2.5 for r in res)      # max over ranks, seen by both
    assert all(r[4] == 129.0 for r in res)


def test_single_process_is_identity():
    assert max_over_ranks(3.25) == 3.25
