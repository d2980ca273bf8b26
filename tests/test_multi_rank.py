"""The N>1 path on CPU with gloo, world size 2.

Decode over a batch shards by sequence with no data-path exchange: each rank
decodes its own contiguous share of the sequences.  Here every rank runs the
oracle on its share; gathering the shares (for the check only) must reproduce the
single-process result.  The benchmark's cross-rank reductions (max of times, sum
of bytes) are checked on the same process group.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from paged_kv_decode_mapping_gb300 import workloads as W

        w = W.small_workload(B=5, Hq=8, Hkv=2, D=16, BS=4, lens=(3, 9, 17, 1, 30), seed=31)
        inp = W.make_inputs(w)
        lo, hi = W.shard_range(w.B, rank, world)
        orc = oracle.get()
        mine = orc.decode(inp["q"][lo:hi], inp["k_cache"], inp["v_cache"],
                          inp["block_tables"][lo:hi], inp["context_lens"][lo:hi], inp["scale"])
        shards = [None] * world
        dist.all_gather_object(shards, (lo, hi, mine))
        t_max = bench.reduce_max(1.0 + rank, world, torch.device("cpu"))
        b_sum = bench.reduce_sum(10.0 * (rank + 1), world, torch.device("cpu"))
        if rank == 0:
            full = orc.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                              inp["context_lens"], inp["scale"])
            got = torch.cat([s[2] for s in sorted(shards, key=lambda s: s[0])])
            q.put((torch.equal(got, full), t_max, b_sum))
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_sequences_without_exchange():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    same, t_max, b_sum = q.get(timeout=10)
    assert same
    assert t_max == 2.0 and b_sum == 30.0
