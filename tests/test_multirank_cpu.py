"""The multi-GPU logic on CPU ranks (gloo, world size 2): the path shards by
request with no collective on the data path (each rank is a replica with its
own pool and request shard), so the only cross-rank steps are the barrier,
the max over ranks of the step time and the sum of the tokens processed.
Also checks that each rank draws its own request shard, and that each rank's
copy of the library validates its own shard's arguments on the host."""
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


def _lib_worker(rank, world, port, q):
    """Each rank loads the library and runs its host-side argument checks on
    a pool descriptor and batch of its own (fake device pointers: nothing is
    enqueued), then the ranks agree on the outcome with one all-reduce."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch

    import __graft_entry__

    if rank == 0:  # one rank compiles; the other finds the library up to date
        __graft_entry__.build()
    dist.barrier()
    __graft_entry__.build()
    import bench
    import paged_fp8_kv_append_gb300 as kv
    import workloads as wl

    w = wl.gqa_batch(seed=bench.shard_seed(20262, rank))
    d = kv.kv_pool_desc()
    d.num_pages, d.page_size, d.num_kv_heads = w.num_pages, w.page_size, w.num_kv_heads
    d.head_dim_k, d.head_dim_v = w.head_dim_k, w.head_dim_v
    d.dtype, d.layout = kv.KV_DTYPE_E4M3, kv.KV_LAYOUT_GQA
    fake = 0x10000 * (rank + 1)  # 16-byte aligned, never dereferenced
    d.k_cache = d.v_cache = d.k_scale = d.v_scale = d.tags = d.free_list = d.ctl = fake
    h = kv.kv_pool_create(d)
    lib = kv._lib
    B = w.B
    checks = [
        lib.kv_append_quantize(h, None, -1, None, None, None, 0, None, None, 4, None) == 1,
        lib.kv_verify_tags(h, None, B, None, None, w.max_pages, None, None) == 1,
        lib.paged_decode_attn(h, None, B, w.num_q_heads, 1, None, None, w.max_pages, None, None,
                              1.0, None, None, 0) == 1,
        lib.paged_decode_attn_checked(h, None, B, w.num_q_heads, 1, fake, fake, None,
                                      w.max_pages, fake, 1.0, fake, fake, fake, 1 << 30) == 1,
        lib.kv_verify_tags(h, None, 0, None, None, w.max_pages, None, None) == 0,
    ]
    # an unaligned cache pointer is refused at pool creation on every rank
    d.k_cache = fake + 8
    try:
        kv.kv_pool_create(d)
        checks.append(False)
    except kv.KVError as e:
        checks.append(e.status == kv.KV_ERR_INVALID_ARG)
    kv.kv_pool_destroy(h)
    ok = torch.tensor([1.0 if all(checks) else 0.0])
    dist.all_reduce(ok, op=dist.ReduceOp.MIN)
    q.put((rank, [bool(c) for c in checks], float(ok.item()), B))
    dist.destroy_process_group()


def test_two_rank_library_argument_checks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_lib_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, checks, agreed, B in res:
        assert all(checks), (rank, checks)
        assert agreed == 1.0 and B == 32
