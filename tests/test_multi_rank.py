"""The N>1 path on CPU with gloo, world size 2.

The store shards by request and the gather by sequence with no exchange
step: each rank's share writes a disjoint set of cache bytes / output rows,
and the union of the shares equals the single-process result.  The
benchmark's cross-rank reductions (max time, summed bytes) and the
reference arm's rank-0-only rule are exercised on the same ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(WORLD),
                      LOCAL_RANK=str(rank))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        import bench
        import oracle
        from paged_quantized_kv_gb300 import workloads as W
        from tests.test_oracle_gather import run_gather
        from tests.test_oracle_store import run_store

        o = oracle.get()
        # --- store, sharded by request --------------------------------------
        full = W.make_store("mr", 3, 64, 2, 64, 16, 16, slots="runs",
                            request_len=16)
        mine = W.shard_store(full, rank, WORLD, unit_tokens=16)
        part = run_store(o, mine)
        parts = [None] * WORLD
        dist.all_gather_object(parts, part)
        # --- gather, sharded by sequence ------------------------------------
        g = W.make_gather("mrg", 4, [7, 64, 1, 90, 33], 16, 32, 40)
        gs, first = W.shard_gather(g, rank, WORLD)
        k, s = run_gather(o, gs)
        gparts = [None] * WORLD
        dist.all_gather_object(gparts, (first, gs.total_tokens, k, s))
        # --- benchmark reductions -------------------------------------------
        mx = bench.max_over_ranks(1.5 + rank, WORLD)
        sm = bench.sum_over_ranks(10.0 * (rank + 1), WORLD)
        seeds = [None] * WORLD
        dist.all_gather_object(seeds, bench.rank_seed(4, rank))
        if rank == 1:
            # the reference arm does nothing on ranks other than 0
            assert bench.run_reference(None) is None
        if rank == 0:
            want = run_store(o, full)
            got = np.full_like(want, 0xAA)
            for p in parts:
                touched = p != 0xAA
                assert not (touched & (got != 0xAA)).any()  # disjoint
                got[touched] = p[touched]
            assert np.array_equal(got, want)
            wk, ws = run_gather(o, g)
            D = g.head_dim
            for first_row, n, kk, ss in gparts:
                assert np.array_equal(kk[: n * D],
                                      wk[first_row * D:(first_row + n) * D])
                assert np.array_equal(ss[: n * 4],
                                      ws[first_row * 4:(first_row + n) * 4])
            assert mx == 2.5 and sm == 30.0
            assert len(set(seeds)) == WORLD
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except BaseException as e:  # report to the parent, never hang it
        q.put((rank, repr(e)))
        raise


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q))
             for r in range(WORLD)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=240) for _ in range(WORLD))
    for p in procs:
        p.join(timeout=60)
    assert results == {0: "ok", 1: "ok"}, results
