"""The benchmark's multi-GPU logic on CPU ranks (gloo, world size 2): the
path shards by request with no collective on the data path, so the only
cross-rank steps are the barrier, the max over ranks of the step time and the
sum of the tokens processed.  Also checks that each rank draws its own
request shard."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads as wl

    ms = 10.0 + 5.0 * rank                # rank 1 is the slower one
    tokens = 32.0 * (rank + 1)
    bench.barrier()
    mx = bench.reduce_max(ms)
    tot = bench.reduce_sum(tokens)
    w = wl.gqa_batch(seed=bench.shard_seed(20262, rank))
    q.put((rank, mx, tot, w.lens.tolist()))
    dist.destroy_process_group()


def test_two_rank_reductions_and_shards():
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
    (r0, mx0, tot0, lens0), (r1, mx1, tot1, lens1) = res
    assert mx0 == mx1 == 15.0          # the step time is the slowest rank's
    assert tot0 == tot1 == 96.0        # tokens of all ranks are summed
    assert lens0 != lens1              # each rank serves its own shard of requests
    assert len(lens0) == len(lens1) == 32
