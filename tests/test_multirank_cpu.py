"""The bench's multi-rank bookkeeping on CPU with gloo, world size 2: every
rank runs its own batch (seed + rank) and the whole-job figures are the
slowest rank's time and the sum of all ranks' bytes."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_122_gb300 import metrics as M
from paged_kv_cache_122_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.get("l3-8b", 0 + rank)
    step_bytes = float(M.useful_bytes(w)["step"])
    dev_ms, e2e_ms = 1.0 + rank, 3.0 - rank
    res = bench.aggregate_over_ranks(dev_ms, e2e_ms, step_bytes, "cpu")
    out[rank] = (res, step_bytes, int(w.seq_lens.sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_with_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    (r0, b0, t0), (r1, b1, t1) = res[0], res[1]
    assert r0 == r1                                  # every rank sees the same whole-job numbers
    assert r0[0] == 2.0 and r0[1] == 3.0             # slowest rank's device and e2e times
    assert r0[2] == b0 + b1                          # bytes of both batches
    assert t0 != t1                                  # each rank ran its own batch
