"""GPU parity of the vocabulary-parallel verify walk (eagle_verify_accept_sharded).

Every target and draft row is split by vocabulary into S shards, each in its own
device buffer, as a vocabulary-parallel LM head leaves it; on the GPU each rank is one
CTA of the sequence's cluster and reads only its shard.  The outputs are compared with
the single-process oracle walk on the whole rows (bit-exact at T = 0, near-ties only
at T = 1) and, at T = 1, with the oracle's CPU-rank protocol (oracle/vocab_parallel.py)
run with one thread per rank, which exchanges exactly at the same four points.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import assert_tie_budget, compare_walks

pytestmark = pytest.mark.gpu


def _cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _tree_case(cfg, B, seed, V, sigma=None):
    trow, drows = W.tree_draft_rows(cfg, seed, B=B, V=V, sigma=sigma)
    tree = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    tgt = W.assemble_target(trow, tree["draft_row"], tree["cand"], cfg.target_std, seed)
    return tgt, drows, tree


def _run_sharded(tgt, drows, tree, cuts, D, T, seed):
    import eagle_tree_speculative_gb300 as E
    ts = [_cuda(tgt[:, :, a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    ds = [_cuda(drows[:, :, a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, path, emit = E.eagle_verify_accept_sharded(
        ts, ds, cuts, _cuda(tree["tokens"]), _cuda(tree["parent"]), D, T, seed,
        draft_row=_cuda(tree["draft_row"]), dev_status=st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(), int(st.item())


class _ThreadComm:
    """all_gather among `world` threads of this process (every rank calls it the same
    number of times, as the protocol does)."""

    def __init__(self, world, rank, board, barrier):
        self.world, self.rank, self.board, self.barrier = world, rank, board, barrier

    def all_gather(self, x):
        self.board[self.rank] = np.array(x, np.float64)
        self.barrier.wait()
        out = np.stack(self.board)
        self.barrier.wait()
        return out


def _cpu_ranks(tgt, drows, tree, cuts, D, T, seed):
    """The oracle's CPU-rank walk, one thread per rank; returns rank 0's outputs."""
    from oracle.vocab_parallel import walk_sharded
    world = len(cuts) - 1
    B, _, V = tgt.shape
    board = [None] * world
    barrier = threading.Barrier(world)
    results = [None] * world

    def rank_main(r):
        comm = _ThreadComm(world, r, board, barrier)
        v0, v1 = cuts[r], cuts[r + 1]
        results[r] = [walk_sharded(comm, tgt[b][:, v0:v1], drows[b][:, v0:v1], tree["tokens"][b],
                                   tree["parent"][b], tree["draft_row"][b], v0, V, D, T, seed, b)
                      for b in range(B)]

    th = [threading.Thread(target=rank_main, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for r in range(1, world):
        assert results[r] == results[0]
    acc = np.array([a for a, _, _ in results[0]], np.int32)
    path = np.full((B, D + 1), -1, np.int32)
    emit = np.full((B, D + 1), -1, np.int32)
    for b, (a, p, e) in enumerate(results[0]):
        path[b, :len(p)] = p
        emit[b, :len(e)] = e
    return acc, path, emit


@pytest.mark.parametrize("V,cuts", [
    (1000, [0, 400, 1000]),                    # two uneven shards
    (1000, [0, 333, 334, 1000]),               # three, one a single id; scalar loads
    (32000, [0, 10000, 21000, 32000]),         # three uneven shards, vector loads
    (32000, [0, 4000, 8000, 12000, 16000, 20000, 24000, 28000, 32000]),   # eight
])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_sharded_walk_matches_oracle(V, cuts, T):
    """EAGLE-2 trees (60 nodes, depth 6, top-10), B = 12, against the single-process oracle;
    at T = 1 also against the oracle's CPU-rank protocol with the same cuts."""
    cfg = W.CONFIGS["eagle2_b1"]
    tgt, drows, tree = _tree_case(cfg, 12, seed=5, V=V)
    acc, path, emit, st = _run_sharded(tgt, drows, tree, cuts, cfg.depth, T, 23)
    assert st == 0
    ref = oracle.verify_accept(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, T, 23,
                               draft_row=tree["draft_row"])
    assert (ref["status"] == 0).all()
    dec, ties = compare_walks(ref, acc, path, emit, exact=(T == 0.0),
                              rows=(tgt, drows, tree["draft_row"], T))
    assert_tie_budget(dec, ties)
    if T > 0:
        ra, rp, re = _cpu_ranks(tgt, drows, tree, cuts, cfg.depth, T, 23)
        # the CPU ranks reproduce the single-process oracle (tests/test_vocab_parallel_cpu.py)
        assert np.array_equal(ra, ref["accept_len"]) and np.array_equal(re, ref["emit"])
        if ties == 0:
            assert np.array_equal(acc, ra) and np.array_equal(path, rp) and np.array_equal(emit, re)


def test_sharded_walk_llama3_8b_vocab_b64():
    """B = 64 sequences of 60-node depth-8 trees over V = 128256 split into 4 uneven
    shards (as a 4-way vocabulary-parallel head would leave it), T = 1."""
    cfg = W.CONFIGS["eagle3_b64"]
    tgt, drows, tree = _tree_case(cfg, 64, seed=2, V=cfg.V)
    cuts = [0, 32064, 64128, 96192, 128256]
    acc, path, emit, st = _run_sharded(tgt, drows, tree, cuts, cfg.depth, 1.0, 9)
    assert st == 0
    ref = oracle.verify_accept(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0, 9,
                               draft_row=tree["draft_row"])
    dec, ties = compare_walks(ref, acc, path, emit, rows=(tgt, drows, tree["draft_row"], 1.0))
    assert_tie_budget(dec, ties)


def test_sharded_walk_host_errors():
    """Bad shard tables are refused on the host through the C ABI, nothing launched:
    an empty shard, bounds that do not start at 0, more than 8 shards, missing draft
    shards at T > 0."""
    import ctypes

    import eagle_tree_speculative_gb300 as E
    L = E.lib()
    t = torch.zeros(1, 4, 8, device="cuda")
    i = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, 4, dtype=torch.int32, device="cuda")

    def call(cuts, draft=True):
        S = len(cuts) - 1
        ptrs = (ctypes.c_void_p * S)(*([t.data_ptr()] * S))
        beg = (ctypes.c_int32 * (S + 1))(*cuts)
        return L.eagle_verify_accept_sharded(ptrs, ptrs if draft else None, beg, S, None,
                                             i.data_ptr(), i.data_ptr(), 1, 4, cuts[-1], 4, 3, 1.0,
                                             0, out.data_ptr(), out.data_ptr(), out.data_ptr(),
                                             None, None, None)
    assert call([0, 4, 4, 8]) == 2                        # empty shard: EAGLE_ERR_SHAPE
    assert call([1, 8]) == 2                              # does not start at 0
    assert call(list(range(10))) == 2                     # 9 shards
    assert call([0, 4, 8], draft=False) == 1              # T > 0 needs draft shards
    torch.cuda.synchronize()
