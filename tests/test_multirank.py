"""Multi-process host logic on CPU (gloo, world size 2): token rows split
across ranks with no exchange on the data path reproduce the unsharded
result exactly, and the step time reduces to the slowest rank."""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from moe_decode_layer_logits_gb300.sharding import token_shard


def test_token_shard_covers_rows_once():
    for T in [0, 1, 2, 37, 64, 8192]:
        for world in [1, 2, 3, 4, 8]:
            spans = [token_shard(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        token_shard(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import oracle as O
    from moe_decode_layer_logits_gb300.inputs import tail_case
    from moe_decode_layer_logits_gb300.sharding import max_over_ranks, token_shard

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = tail_case(37, 512, 32, 8, seed=40, router=True, weights=False)
        a, b = token_shard(c["T"], rank, world)
        L, _ = O.router_logits(c["x"][a:b], c["w_gate"])
        ids, w, _ = O.topk_route(L.astype(np.float32), c["k"], c["scale"])
        out = O.finalize_add_rmsnorm(c["rows"], c["map"][a:b], w, c["shared"][a:b], None, c["residual"][a:b],
                                     c["gamma"], c["eps"])
        parts = [None] * world
        dist.all_gather_object(parts, (a, b, ids, out["residual_out"], out["normed"]))
        slowest = max_over_ranks(1.0 + rank)
        if rank == 0:
            q.put((parts, slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_row_sharding_matches_unsharded():
    import oracle as O
    from moe_decode_layer_logits_gb300.inputs import tail_case

    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts, slowest = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert slowest == 2.0
    c = tail_case(37, 512, 32, 8, seed=40, router=True, weights=False)
    L, _ = O.router_logits(c["x"], c["w_gate"])
    ids, w, _ = O.topk_route(L.astype(np.float32), c["k"], c["scale"])
    full = O.finalize_add_rmsnorm(c["rows"], c["map"], w, c["shared"], None, c["residual"], c["gamma"], c["eps"])
    got_ids = np.concatenate([p[2] for p in parts])
    got_r = np.concatenate([p[3] for p in parts])
    got_n = np.concatenate([p[4] for p in parts])
    assert [p[:2] for p in parts] == [(0, 19), (19, 37)]
    assert np.array_equal(got_ids, ids)
    assert np.array_equal(got_r, full["residual_out"])
    assert np.array_equal(got_n, full["normed"])
