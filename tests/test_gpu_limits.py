"""GPU parity at the documented limits and for empty batches.

The limits: trees of 64 nodes (the last bit of the ancestor masks) and a chain 63
drafts deep; EAGLE-2 expansion with top_k = 16 over depth 16 (3857 candidates) reranked
to 64 nodes; compaction of a 63-draft accepted path.  Each is compared with the oracle
as the other GPU tests do (exact at T = 0 and for integer work, near-ties only at
T = 1, attention rows to 1e-2).  Empty batches go through the Python binding with
zero-size CUDA tensors, whose data pointers are NULL.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import assert_tie_budget, compare_walks
from tests.test_gpu_attention import _check as attn_check
from tests.test_gpu_expand import _check_given_logits

pytestmark = pytest.mark.gpu


def _E():
    import eagle_tree_speculative_gb300 as E
    return E


def _cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def test_expansion_top16_depth16_reranked_to_64():
    """top_k = 16 and depth = 16 (both limits): 1 + 16 + 15 * 256 = 3857 candidates,
    241 draft rows per sequence, reranked to the 64-node maximum."""
    B, k, D, n_out, V = 3, 16, 16, 64, 1000
    R = oracle.draft_rows(k, D)
    drows = (W.per_seq_normal(B, (R, V), 2.0, 81, W.TAG_TARGET) +
             W.per_seq_normal(B, (R, V), 0.5, 81, W.TAG_DRAFT_NOISE)).astype(np.float32)
    _check_given_logits(drows, k, D, n_out)


def _sibling_rank_tokens(drf, par):
    """Each node's token is the draft's r-th choice after its parent, r = the number of
    earlier siblings: distinct siblings, most of them likely under the target."""
    B, n = par.shape
    tok = np.full((B, n), -1, np.int32)
    for b in range(B):
        order = {}
        for i in range(1, n):
            p = int(par[b, i])
            if p not in order:
                order[p] = [np.argsort(-drf[b, p], kind="stable"), 0]
            tok[b, i] = order[p][0][order[p][1]]
            order[p][1] += 1
    return tok


@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("shape", ["chain63", "bushy"])
def test_verify_64_node_trees(shape, T):
    """64 nodes (the limit): a chain of 63 drafts (max_depth 63; sequence 0's draft
    equals its target, so its walk accepts all 63) and random trees of depth <= 16;
    V = 1003 (the scalar-load path), B = 24."""
    E = _E()
    B, n, V = 24, 64, 1003
    tgt = W.per_seq_normal(B, (n, V), 2.0, 83, W.TAG_TARGET)
    drf = (tgt + W.per_seq_normal(B, (n, V), 0.3, 83, W.TAG_DRAFT_NOISE)).astype(np.float32)
    if shape == "chain63":
        par, D = np.broadcast_to(W.chain_tree(n), (B, n)).copy(), n - 1
        drf[0] = tgt[0]                           # draft = target: all 63 drafts accepted
    else:
        par, D = np.stack([W.random_tree(n, 16, 83, b) for b in range(B)]), 16
    tok = _sibling_rank_tokens(drf, par)
    ref = oracle.verify_accept(tgt, drf, tok, par, D, T, seed=7)
    assert (ref["status"] == 0).all()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, path, emit = E.eagle_verify_accept(_cuda(tgt), _cuda(drf), _cuda(tok), _cuda(par), D, T,
                                            7, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    acc = acc.cpu().numpy()
    dec, ties = compare_walks(ref, acc, path.cpu().numpy(), emit.cpu().numpy(), exact=(T == 0.0),
                              rows=(tgt, drf, None, T))
    assert_tie_budget(dec, ties)
    if shape == "chain63":
        assert acc[0] == n - 1                    # path and emit filled to index 63


def test_attention_64_node_trees():
    """64 nodes (bit 63 of the ancestor masks): a chain and a random tree, 4 query
    heads per kv head (256 rows, two M-tiles per (sequence, kv head))."""
    n = 64
    parent = np.stack([W.chain_tree(n), W.random_tree(n, 12, 85, 1)])
    attn_check(B=2, n=n, Hq=8, Hkv=2, kv_len=[300, 1000], Lmax=1000 + n, seed=85, parent=parent)


def test_compaction_of_64_node_paths():
    """max_depth 63: a fully accepted 64-node chain (every row already in place), a
    41-row path that moves most rows, and a root-only acceptance."""
    E = _E()
    nl, B, Hkv, d, n = 2, 3, 2, 128, 64
    D = n - 1
    kv_len = np.array([100, 37, 5], np.int32)
    Lmax = int(kv_len.max()) + n
    kc, vc = W.kv_cache(nl, B, Hkv, Lmax, d, 87)
    path = np.full((B, D + 1), -1, np.int32)
    path[0] = np.arange(n)
    picks = np.sort(W.rng(87, 1).choice(np.arange(1, n), size=40, replace=False))
    path[1, :41] = np.concatenate([[0], picks])
    path[2, 0] = 0
    acc = np.array([D, 40, 0], np.int32)
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).copy()
    kb, vb, klen = bits(kc), bits(vc), kv_len.copy()
    assert oracle.kv_compact(kb, vb, klen, path, acc, D) == 0
    kg, vg, lg = kc.cuda(), vc.cuda(), _cuda(kv_len)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.eagle_kv_compact(kg, vg, lg, _cuda(path), _cuda(acc), D, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(lg.cpu().numpy(), klen)
    assert np.array_equal(bits(kg), kb) and np.array_equal(bits(vg), vb)


def test_empty_batches_through_the_binding():
    """B = 0 through every call of the binding (zero-size CUDA tensors, NULL data
    pointers): each returns without error or device status and leaves its outputs
    empty."""
    E = _E()
    dev = "cuda"
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    f32 = lambda *s: torch.zeros(*s, device=dev)
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32, device=dev)
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device=dev)
    for T in (0.0, 1.0):
        acc, path, emit = E.eagle_verify_accept(f32(0, 4, 256), f32(0, 4, 256), i32(0, 4),
                                                i32(0, 4), 3, T, 0, dev_status=st)
        assert acc.numel() == 0 and path.shape == (0, 4) and emit.shape == (0, 4)
    out = E.eagle_tree_attn(bf(0, 4, 2, 128), bf(0, 2, 16, 128), bf(0, 2, 16, 128), i32(0),
                            i32(0, 4), dev_status=st)
    assert out.shape == (0, 4, 2, 128)
    out = E.eagle_ttt_attn(bf(0, 8, 4, 128), bf(0, 2, 3, 8, 128), bf(0, 2, 3, 8, 128), 1,
                           dev_status=st)
    assert out.shape == (0, 8, 4, 128)
    E.eagle_kv_compact(bf(1, 0, 2, 16, 128), bf(1, 0, 2, 16, 128), i32(0), i32(0, 4), i32(0), 3,
                       dev_status=st)
    k, D, n_out = 10, 3, 20
    state = torch.zeros(max(1, E.tree_state_size(0, k, D)), dtype=torch.uint8, device=dev)
    for lvl in range(1, D + 1):
        E.eagle2_expand(lvl, lvl == D, f32(0, oracle.draft_rows(k, D), 100), k, D, n_out, state,
                        out_tokens=i32(0, n_out), out_parent=i32(0, n_out),
                        out_draft_row=i32(0, n_out), dev_status=st)
    cand = E.eagle2_tree_candidates(state, 0, k, D)
    assert all(t.numel() == 0 for t in cand.values())
    gm, gz, ga = E.eagle_softmax_stats(f32(0, 100), 1.0, dev_status=st)
    assert gm.numel() == 0 and gz.numel() == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
