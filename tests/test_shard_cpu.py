"""The sharded path's host logic on CPU: shard bounds, and the exchange of the
per-shard totals between two ranks over gloo.

Each rank takes its shard of the array (partition_pass_tile_gb300.shard.
shard_bounds), computes its shard's total with the oracle (the GPU path uses
gc_reduce / gc_count_if), and exchanges it with shard.gather_totals, the same
all-gather the GPU path runs over NCCL.  From the gathered totals each rank
takes its offsets as the oracle's exclusive scan of them (what
gc_shard_offsets computes on the device, tested on the GPU in
tests/test_shard_gpu.py), places its piece with the oracle, and rank 0
checks that the pieces assemble into the oracle's answer for the whole array:
the scan (carry + local scan), the select-if (survivors at base), and the
stable partition (kept at kept-before, rejected at T + start - kept-before).
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_the_array():
    sys.path.insert(0, ROOT)
    from partition_pass_tile_gb300 import shard
    for n in (0, 1, 7, 100, 100_003):
        for parts in (1, 2, 3, 8):
            b = [shard.shard_bounds(n, parts, r) for r in range(parts)]
            assert b[0][0] == 0 and b[-1][1] == n
            assert all(b[r][1] == b[r + 1][0] for r in range(parts - 1))
            sizes = shard.shard_sizes(n, parts)
            assert sum(sizes) == n and max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.shard_bounds(10, 2, 2)


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        from partition_pass_tile_gb300 import shard, synth
        orc = O.default()
        n = 100_003
        a, b = shard.shard_bounds(n, world, rank)
        res = {}

        def exchange(value):
            got = shard.gather_totals(torch.tensor([value], dtype=torch.int32))
            return got.numpy().view(np.uint32)

        # scan: carry = exclusive scan of the shard totals
        x = synth.uniform_i32(n, 21)
        local = x[a:b]
        scan, total = orc.exclusive_scan(local)
        totals = exchange(np.uint32(total).view(np.int32))
        carry = orc.exclusive_scan(totals)[0][rank]
        res["scan"] = (a, (scan.view(np.uint32) + np.uint32(carry)).view(np.int32))
        # select-if: survivors at base = exclusive scan of the shard counts
        y = synth.keep_fraction(n, 0.3, 22)
        kept = orc.select_if(y[a:b], O.NONZERO)
        counts = exchange(kept.shape[0])
        base = int(orc.exclusive_scan(counts)[0][rank])
        res["select"] = (base, kept, int(counts.sum()))
        # partition: kept at kept-before, rejected at T + start - kept-before
        z = synth.uniform_i32(n, 23)
        parted, t = orc.partition(z[a:b], O.EVEN)
        counts = exchange(t)
        kb = int(orc.exclusive_scan(counts)[0][rank])
        T = int(counts.sum())
        res["partition"] = (kb, parted[:t], T + a - kb, parted[t:])
        pieces = [None] * world
        dist.all_gather_object(pieces, res)
        if rank == 0:
            ok = {}
            whole = np.empty(n, dtype=np.int32)
            for p in pieces:
                s0, v = p["scan"]
                whole[s0:s0 + v.shape[0]] = v
            ok["scan"] = np.array_equal(whole, orc.exclusive_scan(x)[0])
            want = orc.select_if(y, O.NONZERO)
            got = np.full(pieces[0]["select"][2], -1, dtype=np.int32)
            for p in pieces:
                s0, v, _ = p["select"]
                got[s0:s0 + v.shape[0]] = v
            ok["select"] = np.array_equal(got, want)
            wantp, wt = orc.partition(z, O.EVEN)
            gotp = np.full(n, -1, dtype=np.int32)
            for p in pieces:
                k0, kv, r0, rv = p["partition"]
                gotp[k0:k0 + kv.shape[0]] = kv
                gotp[r0:r0 + rv.shape[0]] = rv
            ok["partition"] = np.array_equal(gotp, wantp)
            q.put(ok)
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_totals_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    ok = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok == {"scan": True, "select": True, "partition": True}
