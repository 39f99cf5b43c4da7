"""Multi-rank path on the CPU: two gloo ranks, each running half of the heads.

The (batch, head) pairs are independent, so the half-head shards must
reproduce the single-process result exactly, and the timing reduction must
return the slowest rank's time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from kv_cache_eviction_03_gb300 import sharding
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

W_TINY = W.Workload("shard", 1, 4, 16, "f32", 40, 8, 6, 5, 1.1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run_heads(lo, hi):
    w = W_TINY
    q, k, v = W.prefill_inputs(w, 5)
    st, _, _ = O.prefill(q[:, lo:hi], k[:, lo:hi], v[:, lo:hi], w.heavy, w.recent, w.scale)
    outs = []
    for t in range(w.decode):
        qd, kd, vd = W.decode_inputs(w, w.prompt + t, 5)
        st, out, _, _ = O.decode_step(st, qd[:, lo:hi], kd[:, lo:hi], vd[:, lo:hi], w.heavy, w.recent, w.scale)
        outs.append(out)
    return np.stack(outs), st.pos


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = sharding.shard_range(W_TINY.heads, world, rank)
        outs, pos = run_heads(lo, hi)
        gathered = [None] * world
        dist.all_gather_object(gathered, (lo, hi, outs, pos))
        slowest = sharding.max_over_ranks([float(rank + 1), -float(rank)], dist)
        if rank == 0:
            q.put((gathered, slowest))
    finally:
        dist.destroy_process_group()


def test_shard_range_covers_everything():
    for n in (1, 4, 7, 56, 3584):
        for world in (1, 2, 3, 8):
            parts = [sharding.shard_range(n, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [hi - lo for lo, hi in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharding.shard_range(4, 2, 2)


def test_two_gloo_ranks_reproduce_the_full_run():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, slowest = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full_out, full_pos = run_heads(0, W_TINY.heads)
    out = np.concatenate([g[2] for g in sorted(gathered, key=lambda g: g[0])], axis=1)
    pos = np.concatenate([g[3] for g in sorted(gathered, key=lambda g: g[0])], axis=0)
    assert np.array_equal(out, full_out)
    assert np.array_equal(pos, full_pos)
    assert slowest == [2.0, 0.0]
