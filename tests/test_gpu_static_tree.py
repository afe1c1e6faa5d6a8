"""GPU parity for static draft trees (EAGLE-1 / Medusa style) against the oracle.

The tree is planned from a list of rank paths (choices); each level's tokens are the
ranked tokens of the parent's draft row (bit-exact, ties to the lower token).  The
tree then drives tree attention (its parent array is the mask source) and verify
(its draft_row array names each internal node's draft distribution), both checked
against the oracle with the tolerances of the EAGLE-2 tests.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import assert_tie_budget, attn_row_rel_err, compare_walks

pytestmark = pytest.mark.gpu


def _E():
    import eagle_tree_speculative_gb300 as E
    return E


def _choices(seed, cap, width):
    """A prefix-closed random choice set: breadth-first growth, up to `width` children."""
    g = W.rng(seed, 50)
    choices, frontier = [], [()]
    while frontier and len(choices) < cap:
        c = frontier.pop(0)
        for r in range(int(g.integers(1, width + 1))):
            if len(choices) < cap:
                choices.append(c + (r,))
                frontier.append(c + (r,))
    return choices


def _tokens_gpu(tree, logits):
    E = _E()
    B, R, V = logits.shape
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in tree.items()}
    n = len(tree["parent"])
    tok = torch.full((B, n), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    for level in range(1, int(tree["depth"].max()) + 1):
        E.eagle_static_tree_level(level, lg, dev["parent"], dev["rank"], dev["depth"],
                                  dev["draft_row"], tok, dev_status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("V,cap,width", [(32000, 59, 4), (1001, 40, 6), (128256, 47, 3)])
def test_static_tree_tokens_match_oracle(V, cap, width):
    B = 8
    tree = _E().eagle_static_tree(_choices(V, cap, width))
    R = int(tree["draft_row"].max()) + 1
    logits = W.per_seq_normal(B, (R, V), 2.0, 3, W.TAG_TARGET)
    logits[0, 0, 5] = logits[0, 0, 9] = logits[0, 0].max() + 1.0     # a tie: lower token first
    got, st = _tokens_gpu(tree, logits)
    assert st == 0
    ref = oracle.static_tree_tokens(logits, tree)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_static_tree_verify_and_attention_match_oracle(T):
    """A 60-node static tree, V = 32000, B = 8: tokens, then verify (draft rows = target
    rows + noise, as the EAGLE-2 verify tests) and tree attention on its parent array."""
    E = _E()
    B, V = 8, 32000
    tree = E.eagle_static_tree(_choices(7, 59, 4))
    n = len(tree["parent"])
    R = int(tree["draft_row"].max()) + 1
    trow = W.per_seq_normal(B, (R, V), 2.0, 11, W.TAG_TARGET)
    drows = (trow + W.per_seq_normal(B, (R, V), 0.5, 11, W.TAG_DRAFT_NOISE)).astype(np.float32)
    tok, st = _tokens_gpu(tree, drows)
    assert st == 0 and np.array_equal(tok, oracle.static_tree_tokens(drows, tree))
    drow = np.broadcast_to(tree["draft_row"], (B, n)).copy()
    cand = np.broadcast_to(np.arange(n, dtype=np.int32), (B, n))
    tgt = W.assemble_target(trow, drow, cand, 2.0, 11)
    par = np.broadcast_to(tree["parent"], (B, n)).copy()
    D = int(tree["depth"].max())
    ref = oracle.verify_accept(tgt, drows, tok, par, D, T, seed=3, draft_row=drow)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    acc, path, emit = E.eagle_verify_accept(cu(tgt), cu(drows), cu(tok), cu(par), D, T, 3,
                                            draft_row=cu(drow), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and (ref["status"] == 0).all()
    dec, ties = compare_walks(ref, acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(),
                              exact=(T == 0.0), rows=(tgt, drows, drow, T))
    assert_tie_budget(dec, ties)
    assert ref["accept_len"].mean() > 0.3
    # tree attention with the static tree as the mask source (Vicuna-like heads, short cache)
    q, k, v, kv_len = W.attn_inputs(2, n, 8, 8, 128, [300, 257], 300 + n, 12)
    out = E.eagle_tree_attn(q.cuda(), k.cuda(), v.cuda(), cu(kv_len), cu(par[:2]), scale=128 ** -0.5,
                            dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.float().cpu().numpy()
    for b in range(2):
        r = oracle.tree_attn(q[b:b + 1], k[b:b + 1], v[b:b + 1], kv_len[b:b + 1], par[b:b + 1],
                             128 ** -0.5)
        assert attn_row_rel_err(got[b:b + 1], r).max() <= 1e-2
