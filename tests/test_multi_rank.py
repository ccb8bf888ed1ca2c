"""World-size-2 gloo tests (CPU) of the multi-GPU host logic.

Each rank takes its block of output rows of the same layer, runs the CPU
oracle's search on that block, and the ranks combine their per-alpha block
losses with one all-reduce; the result must equal the oracle's search over
the whole layer. The timing reduction must return the slowest rank.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
import workloads
from post_bit_weight_awq_b300 import multi


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_features, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = workloads.make_layer("llama7b_q_proj", n_tok=96, out_features=out_features, in_features=256)
        X = L["X"].astype(np.float64)
        sx = O.channel_importance(X)
        r0, r1 = multi.shard_rows(out_features, world, rank)
        res = O.search_scale(L["W"][r0:r1].astype(np.float64), X, sx)
        losses, best = multi.combine_row_shards(res["losses"], X.shape[0], r1 - r0, out_features)
        t = multi.max_over_ranks(1.0 + rank)
        q.put((rank, losses, best, t, (r0, r1)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("out_features", [64, 37])
def test_row_sharded_search_equals_whole_layer(out_features):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out_features, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    L = workloads.make_layer("llama7b_q_proj", n_tok=96, out_features=out_features, in_features=256)
    full = O.search_scale(L["W"].astype(np.float64), L["X"].astype(np.float64), O.channel_importance(L["X"]))
    spans = [r[4] for r in results]
    assert spans[0][0] == 0 and spans[0][1] == spans[1][0] and spans[1][1] == out_features
    for rank, losses, best, t, _ in results:
        np.testing.assert_allclose(losses, full["losses"], rtol=1e-12)
        assert best == full["best_idx"]
        assert t == 2.0  # slowest rank


def test_shard_rows_cover_every_row_once():
    for out in (1, 7, 4096, 11008):
        for world in (1, 2, 3, 8):
            spans = [multi.shard_rows(out, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == out
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
