"""The multi-GPU bench path on CPU: world_size-2 gloo process groups.

Decode shards by sequence with no exchange, so N GPUs run N independent
replicas.  The only cross-rank steps are the barrier and the reduction of the
timed region (slowest rank's time, sum of every rank's work); these run here
with the gloo backend, ranks launched as separate processes on 127.0.0.1.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_102_gb300 import workloads as W
    try:
        dist, r, ws, local = bench._dist()  # gloo: no CUDA here
        assert (r, ws, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        # each rank draws its own batch (seed + rank), as the bench does
        wl = W.WORKLOADS["llama7b"]
        lens = W.draw(wl, 7 + rank).context_lens + 1
        dec, app = bench.algorithmic_bytes(wl, lens)
        seconds = [0.010, 0.025][rank]
        t, job = bench.reduce_over_ranks(dist, torch.device("cpu"), seconds, {"bytes": dec + app, "seqs": len(lens)})
        dist.barrier()
        q.put((rank, t, job, dec + app, len(lens), int(lens.sum())))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, repr(e)))


def test_replicas_reduce_time_max_and_work_sum():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for res in results:
        assert len(res) == 6, f"rank {res[0]} failed: {res[1]}"
    results.sort()
    total_bytes = sum(r[3] for r in results)
    total_seqs = sum(r[4] for r in results)
    for rank, t, job, *_ in results:
        assert t == pytest.approx(0.025)          # the slowest rank's time
        assert job["bytes"] == pytest.approx(total_bytes)
        assert job["seqs"] == total_seqs
    # the ranks drew different batches, so their work differs
    assert results[0][5] != results[1][5]


def test_reduce_without_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    t, job = bench.reduce_over_ranks(None, torch.device("cpu"), 1.5, {"bytes": 10, "seqs": 3})
    assert t == 1.5 and job == {"bytes": 10.0, "seqs": 3.0}
