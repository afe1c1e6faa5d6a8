"""Vocab-parallel verify on CPU ranks: the walk with the vocabulary split across 2 or 3
gloo ranks (oracle/vocab_parallel.py) equals the single-process oracle walk.

Each rank holds a slice of every target and draft row and exchanges only what the
walk needs: row statistics, the drafted token's probabilities, residual normalisers
and the race winners.  Same seeded inputs on every rank; decisions must agree except
near-ties; in fp64 none occurs on these inputs, so the outputs must be identical.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _Comm:
    def __init__(self, world):
        self.world = world

    def all_gather(self, x):
        t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, np.float64)))
        out = [torch.empty_like(t) for _ in range(self.world)]
        dist.all_gather(out, t)
        return np.stack([o.numpy() for o in out])


def _case(V=1000, B=12, seed=5):
    cfg = W.CONFIGS["eagle2_b1"]
    trow, drows = W.tree_draft_rows(cfg, seed, B=B, V=V)
    tree = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    tgt = W.assemble_target(trow, tree["draft_row"], tree["cand"], cfg.target_std, seed)
    return cfg, tgt, drows, tree


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle.vocab_parallel import walk_sharded
        cfg, tgt, drows, tree = _case()
        V = tgt.shape[-1]
        cuts = [0, 400, 1000] if world == 2 else [0, 333, 334, 1000]     # uneven slices
        v0, v1 = cuts[rank], cuts[rank + 1]
        comm = _Comm(world)
        res = []
        for b in range(tgt.shape[0]):
            res.append(walk_sharded(comm, tgt[b][:, v0:v1], drows[b][:, v0:v1], tree["tokens"][b],
                                    tree["parent"][b], tree["draft_row"][b], v0, V, cfg.depth,
                                    1.0, 23, b))
        out[rank] = res
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_walk_equals_single_process_walk(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    cfg, tgt, drows, tree = _case()
    ref = oracle.verify_accept(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0, 23,
                               draft_row=tree["draft_row"])
    assert (ref["status"] == 0).all()
    for r in range(1, world):                       # every rank reaches the same result
        assert res[r] == res[0]
    mism = 0
    for b, (a, path, emit) in enumerate(res[0]):
        ra = int(ref["accept_len"][b])
        same = (a == ra and path == ref["path"][b, :ra + 1].tolist()
                and emit == ref["emit"][b, :ra + 1].tolist())
        mism += not same
    assert mism == 0, mism
    assert ref["accept_len"].mean() > 0.5
