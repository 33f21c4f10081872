"""Multi-rank bench logic on CPU with the gloo backend, world size 2: each
rank owns an independent batch of heads (weak scaling, disjoint ranges and
seeds), and the timed region's duration is reduced with a max over ranks.
No data-path collective exists; only this timing reduction and barriers."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    seed, heads = bench.shard_heads(r, w, 2, 16)
    elapsed = 10.0 + 5.0 * rank          # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, w)
    bench.barrier(w)
    out[rank] = (r, w, local, seed, heads, m)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_shard_heads_and_take_max_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs)
    r0, r1 = out[0], out[1]
    assert (r0[0], r0[1]) == (0, 2) and (r1[0], r1[1]) == (1, 2)
    assert r0[3] != r1[3]                                 # distinct input seeds
    assert r0[4] == (0, 32) and r1[4] == (32, 64)         # disjoint head ranges
    assert r0[5] == r1[5] == 15.0                         # both see the slowest rank's time
