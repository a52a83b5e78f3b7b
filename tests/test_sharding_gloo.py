"""Request sharding across ranks, on the CPU with two gloo ranks.

No step of the path couples two requests, so a batch split by request over
ranks (one replica per GPU, no collective on the data path) must give exactly
the unsharded results.  Each rank corrects its share of a seeded batch with
the oracle; rank 0 gathers the shards and compares them with the whole batch
corrected in one process.  The timing reduction bench.py applies across ranks
(max of the elapsed times) is exercised on the same process group.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

N, V, D, SLOTS, K = 4, 512, 64, 6, 8


def shard(n: int, rank: int, world: int) -> range:
    """Contiguous request ranges, sizes differing by at most one."""
    per, extra = divmod(n, world)
    start = rank * per + min(rank, extra)
    return range(start, start + per + (1 if rank < extra else 0))


def _problem():
    import synth
    import oracle
    rng = np.random.default_rng(2024)
    logits = synth.make_logits(rng, N, SLOTS, V, 8, (4.0, 12.0))
    hidden = synth.make_hidden(rng, N, SLOTS, D)
    E = synth.make_embedding(np.random.default_rng([2024, V, D]), V, D)
    w = synth.make_weights(rng, D, perturb=True)
    model = oracle.Model(w, V=V, d=D, slots=SLOTS, K=K)
    targets = rng.integers(0, V, size=(N, SLOTS - 1)).astype(np.int32)
    return model, logits, hidden, E, targets


def _rank_main(rank: int, world: int, port: int, out: dict):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        model, logits, hidden, E, targets = _problem()
        mine = list(shard(N, rank, world))
        res = oracle.correct_batch(model, logits, hidden, E, targets, requests=mine, threads=1)
        tokens = torch.full((N, SLOTS - 1), -1, dtype=torch.int64)
        accept = torch.full((N,), -1, dtype=torch.int64)
        scores = torch.zeros((N, SLOTS - 2, K, K), dtype=torch.float64)
        for j, n in enumerate(mine):
            tokens[n] = torch.from_numpy(res["tokens"][j].astype(np.int64))
            accept[n] = int(res["accept_len"][j])
            scores[n] = torch.from_numpy(res["scores"][j])
        # each request is owned by exactly one rank: a sum gathers the shards
        for t in (tokens, accept, scores):
            mask = torch.zeros_like(t)
            for n in mine:
                mask[n] = 1
            t.mul_(mask)
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
        owned = torch.tensor([len(mine)], dtype=torch.int64)
        dist.all_reduce(owned, op=dist.ReduceOp.SUM)
        # bench.py's cross-rank timing reduction
        elapsed = torch.tensor([1.0 + rank], dtype=torch.float64)
        dist.all_reduce(elapsed, op=dist.ReduceOp.MAX)
        if rank == 0:
            out["tokens"] = tokens.numpy().copy()
            out["accept"] = accept.numpy().copy()
            out["scores"] = scores.numpy().copy()
            out["owned"] = int(owned.item())
            out["elapsed"] = float(elapsed.item())
    finally:
        dist.destroy_process_group()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2])
def test_request_sharding_matches_unsharded(world):
    import oracle
    oracle.build()
    assert [len(shard(N, r, world)) for r in range(world)] == [2, 2]
    assert sorted(n for r in range(3) for n in shard(7, r, 3)) == list(range(7))
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(out)
    model, logits, hidden, E, targets = _problem()
    ref = oracle.correct_batch(model, logits, hidden, E, targets, threads=1)
    assert got["owned"] == N
    assert got["elapsed"] == float(world)
    np.testing.assert_array_equal(got["tokens"], ref["tokens"].astype(np.int64))
    np.testing.assert_array_equal(got["accept"], np.asarray(ref["accept_len"], dtype=np.int64))
    np.testing.assert_array_equal(got["scores"], ref["scores"])
