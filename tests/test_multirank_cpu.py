"""The N > 1 host logic on CPU with two gloo ranks (no GPU).

Each rank owns a disjoint token range or its own seeded batch; the only
collectives are the barrier and the max/sum reductions of the timing.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

from sparse_mla_attention_token_gb300 import dist as sdist


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    assert sdist.init("gloo")
    sdist.barrier()
    r, lr, w = sdist.env_world()
    mx = sdist.max_over_ranks(1.5 + r)
    sm = sdist.sum_over_ranks(10.0 * (r + 1))
    rng = sdist.shard_range(4097, r, w)
    q.put((r, mx, sm, rng, sdist.rank_seed(3, r)))
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
    assert [x[1] for x in res] == [2.5, 2.5]
    assert [x[2] for x in res] == [30.0, 30.0]
    (a0, b0), (a1, b1) = res[0][3], res[1][3]
    assert a0 == 0 and b0 == a1 and b1 == 4097
    assert res[0][4] != res[1][4]


@pytest.mark.parametrize("n,world", [(10, 3), (4096, 8), (5, 8), (0, 2)])
def test_shard_range_covers_once(n, world):
    got = [sdist.shard_range(n, r, world) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == n
    for (a, b), (c, d) in zip(got, got[1:]):
        assert b == c and b - a >= d - c and (b - a) - (d - c) <= 1


def test_single_process_identity():
    assert sdist.max_over_ranks(3.25) == 3.25
    if "WORLD_SIZE" not in os.environ:
        assert sdist.init("gloo") is False
