"""GPU parity of eagle_verify_accept and eagle_softmax_stats against the oracle.

Same seeded inputs on both sides (workloads/), element-by-element comparison:
bit-exact at temperature 0; at temperature 1 identical except counted
near-ties (see tests/helpers.py for the tolerances).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import assert_tie_budget, compare_walks

pytestmark = pytest.mark.gpu


def _gpu():
    import eagle_tree_speculative_gb300 as E
    return E


def _cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _run_gpu(tgt, drf, tok, par, D, T, seed, draft_row=None, row_stats=False):
    E = _gpu()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs = None
    if row_stats:
        B, n, _ = tgt.shape
        rs = torch.full((2, B, n, 2), float("nan"), device="cuda")
    acc, path, emit = E.eagle_verify_accept(
        _cuda(tgt), None if drf is None else _cuda(drf), _cuda(tok), _cuda(par), D, T, seed,
        draft_row=None if draft_row is None else _cuda(draft_row), row_stats=rs, dev_status=status)
    torch.cuda.synchronize()
    out = (acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(), int(status.item()))
    return out + ((rs.cpu().numpy(),) if row_stats else ())


# ---------------------------------------------------------------- chain (1000 steps)
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_chain_1000_steps_match_oracle(T):
    cfg = W.CONFIGS["chain"]
    B, n, V, D = 1000, cfg.n, cfg.V, cfg.depth
    tgt, drf = W.chain_logits(B, n, V, cfg.sigma, cfg.target_std, seed=0)
    tok = np.full((B, n), -1, np.int32)
    tok[:, 1:] = oracle.sample_rows(drf[:, :n - 1], T, seed=0)    # draft i+1 ~ p(after node i)
    par = np.broadcast_to(W.chain_tree(n), (B, n)).copy()
    ref = oracle.verify_accept(tgt, drf, tok, par, D, T, seed=0)
    acc, path, emit, st, rs = _run_gpu(tgt, drf, tok, par, D, T, 0, row_stats=True)
    assert st == 0 and (ref["status"] == 0).all()
    dec, ties = compare_walks(ref, acc, path, emit, exact=(T == 0.0), rows=(tgt, drf, None, T))
    assert_tie_budget(dec, ties)
    if T > 0:
        # softmax statistics of every visited row, 1e-5 relative
        m, Z, _, _ = oracle.softmax_rows(tgt, T)
        seen = ~np.isnan(rs[0, :, :, 0])
        assert seen.sum() >= B
        np.testing.assert_allclose(rs[0][..., 0][seen], m[seen], rtol=1e-6)
        np.testing.assert_allclose(rs[0][..., 1][seen], Z[seen], rtol=1e-5)
        mp, Zp, _, _ = oracle.softmax_rows(drf, T)
        seen = ~np.isnan(rs[1, :, :, 0])
        np.testing.assert_allclose(rs[1][..., 1][seen], Zp[seen], rtol=1e-5)


# ---------------------------------------------------------------- EAGLE-2 trees
def _tree_case(cfg, B, seed, V=None, sigma=None):
    V = cfg.V if V is None else V
    trow, drows = W.tree_draft_rows(cfg, seed, B=B, V=V, sigma=sigma)
    tree = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    tgt = W.assemble_target(trow, tree["draft_row"], tree["cand"], cfg.target_std, seed)
    return tgt, drows, tree


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_eagle2_tree_b1_shape_matches_oracle(T):
    cfg = W.CONFIGS["eagle2_b1"]
    B = 40                                     # 40 independent B=1 problems in one launch
    tgt, drows, tree = _tree_case(cfg, B, seed=1)
    ref = oracle.verify_accept(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, T, seed=5,
                               draft_row=tree["draft_row"])
    acc, path, emit, st = _run_gpu(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, T, 5,
                                   draft_row=tree["draft_row"])
    assert st == 0
    dec, ties = compare_walks(ref, acc, path, emit, exact=(T == 0.0),
                              rows=(tgt, drows, tree["draft_row"], T))
    assert_tie_budget(dec, ties)
    assert ref["accept_len"].mean() > 0.5     # the synthetic draft is informative


@pytest.mark.parametrize("V,T,sigma", [(32000, 0.0, 0.5), (32000, 1.0, 0.5), (128256, 0.0, 0.5),
                                         (128256, 1.0, 0.5), (32000, 1.0, 0.1), (32000, 1.0, 1.0)])
def test_llama70b_sweep_trees_match_oracle(V, T, sigma):
    """Sweep shape: 48-node depth-6 top-10 trees, B=8, across vocabulary, temperature
    and draft noise (sigma sets how often the draft is accepted)."""
    cfg = W.CONFIGS["sweep_70b"]
    tgt, drows, tree = _tree_case(cfg, 8, seed=31, V=V, sigma=sigma)
    ref = oracle.verify_accept(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, T, seed=13,
                               draft_row=tree["draft_row"])
    acc, path, emit, st = _run_gpu(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, T, 13,
                                   draft_row=tree["draft_row"])
    assert st == 0 and (ref["status"] == 0).all()
    dec, ties = compare_walks(ref, acc, path, emit, exact=(T == 0.0),
                              rows=(tgt, drows, tree["draft_row"], T))
    assert_tie_budget(dec, ties)


@pytest.fixture(scope="module",
                params=[(V, sg) for V in (32000, 128256) for sg in (0.1, 0.5, 1.0)],
                ids=lambda p: f"V{p[0]}-sigma{p[1]}")
def sweep_b64(request):
    """Llama-70B sweep trees (48 nodes, depth 6, top-10) for 64 sequences at one (V, sigma);
    the first 32 sequences are the B = 32 case (inputs are keyed per sequence)."""
    V, sigma = request.param
    tgt, drows, tree = _tree_case(W.CONFIGS["sweep_70b"], 64, seed=71, V=V, sigma=sigma)
    return V, sigma, tgt, drows, tree


@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("B", [32, 64])
def test_llama70b_sweep_full_batches_match_oracle(sweep_b64, B, T):
    """The sweep's verify at B = 32 and 64, V in {32000, 128256}, T in {0, 1}, draft noise
    sigma in {0.1, 0.5, 1.0}: bit-exact at T = 0, near-ties only at T = 1."""
    V, sigma, tgt, drows, tree = sweep_b64
    cfg = W.CONFIGS["sweep_70b"]
    t, d = tgt[:B], drows[:B]
    tk, pa, dr = tree["tokens"][:B], tree["parent"][:B], tree["draft_row"][:B]
    ref = oracle.verify_accept(t, d, tk, pa, cfg.depth, T, seed=19, draft_row=dr)
    acc, path, emit, st = _run_gpu(t, d, tk, pa, cfg.depth, T, 19, draft_row=dr)
    assert st == 0 and (ref["status"] == 0).all()
    dec, ties = compare_walks(ref, acc, path, emit, exact=(T == 0.0), rows=(t, d, dr, T))
    assert_tie_budget(dec, ties)
    print(f"B={B} V={V} T={T} sigma={sigma}: mean accept_len {ref['accept_len'].mean():.3f}, "
          f"decisions {dec}, near-ties {ties}")


def test_eagle3_tree_b64_full_size_matches_oracle():
    """Full B=64, n=60, depth 8, V=128256 verify (sigma 0.3, T=1)."""
    cfg = W.CONFIGS["eagle3_b64"]
    tgt, drows, tree = _tree_case(cfg, cfg.B, seed=2)
    ref = oracle.verify_accept(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0, seed=9,
                               draft_row=tree["draft_row"])
    acc, path, emit, st = _run_gpu(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0, 9,
                                   draft_row=tree["draft_row"])
    assert st == 0
    dec, ties = compare_walks(ref, acc, path, emit, rows=(tgt, drows, tree["draft_row"], 1.0))
    assert_tie_budget(dec, ties)


@pytest.mark.parametrize("V", [1001, 7])
def test_unaligned_vocab_and_tiny_vocab(V):
    """V not a multiple of 4 takes the scalar path; V=7 leaves some CTAs of a cluster empty."""
    B, n = 33, 9
    tgt = W.per_seq_normal(B, (n, V), 2.0, 4, W.TAG_TARGET)
    drf = tgt + W.per_seq_normal(B, (n, V), 0.7, 4, W.TAG_DRAFT_NOISE)
    par = np.stack([W.random_tree(n, 4, 4, b) for b in range(B)])
    tok = W.rng(4, 5).integers(0, V, size=(B, n), dtype=np.int32)
    for T in (1.0, 0.0):
        ref = oracle.verify_accept(tgt, drf, tok, par, 4, T, seed=3)
        acc, path, emit, st = _run_gpu(tgt, drf, tok, par, 4, T, 3)
        assert st == 0
        dec, ties = compare_walks(ref, acc, path, emit, exact=(T == 0.0), rows=(tgt, drf, None, T))
        assert_tie_budget(dec, ties)


def test_root_only_tree_emits_one_bonus_token():
    B, V = 50, 500
    tgt = W.per_seq_normal(B, (1, V), 2.0, 6, W.TAG_TARGET)
    par = np.full((B, 1), -1, np.int32)
    tok = np.full((B, 1), -1, np.int32)
    ref = oracle.verify_accept(tgt, tgt, tok, par, 0, 1.0, seed=8)
    acc, path, emit, st = _run_gpu(tgt, tgt, tok, par, 0, 1.0, 8)
    assert st == 0 and (acc == 0).all() and (path[:, 0] == 0).all()
    compare_walks(ref, acc, path, emit, rows=(tgt, tgt, None, 1.0))


def test_device_errors_flag_and_skip_without_trapping():
    E = _gpu()
    V, n = 64, 4
    tgt = W.per_seq_normal(4, (n, V), 1.0, 7, W.TAG_TARGET)
    tgt[3, 0, 5] = np.nan
    par = np.array([[-1, 0, 1, 2], [-1, 0, 3, 1], [0, 0, 1, 2], [-1, 0, 0, 1]], np.int32)
    tok = np.array([[-1, 1, 2, 3], [-1, 1, 2, 3], [-1, 1, 2, 3], [-1, 1, 2, 3]], np.int32)
    tok[0, 2] = V                                             # token out of range
    acc, path, emit, st = _run_gpu(tgt, tgt, tok, par, 3, 1.0, 0)
    assert list(acc) == [-1, -1, -1, -1]
    assert st & E.EAGLE_DEV_BAD_TREE and st & E.EAGLE_DEV_BAD_TOKEN and st & E.EAGLE_DEV_NONFINITE
    assert (path == -1).all() and (emit == -1).all()
    # the context is healthy afterwards
    tok[0, 2] = 2
    par[1], par[2] = par[0], par[0]
    tgt[3, 0, 5] = 0.0
    acc, path, emit, st = _run_gpu(tgt, tgt, tok, par, 3, 1.0, 0)
    assert st == 0 and (acc >= 0).all()


def test_host_side_validation_returns_status_without_launch():
    E = _gpu()
    t = torch.zeros(1, 65, 8, device="cuda")
    i = torch.zeros(1, 65, dtype=torch.int32, device="cuda")
    with pytest.raises(E.EagleError) as ex:
        E.eagle_verify_accept(t, t, i, i, 3, 1.0, 0)
    assert ex.value.code == 2                                 # n > 64 -> EAGLE_ERR_SHAPE
    with pytest.raises(E.EagleError) as ex:
        E.eagle_verify_accept(t[:, :4], t[:, :4], i[:, :4], i[:, :4], 3, -1.0, 0)
    assert ex.value.code == 1                                 # T < 0


# ---------------------------------------------------------------- softmax statistics
@pytest.mark.parametrize("V,T", [(32000, 1.0), (1001, 0.7), (32000, 0.0)])
def test_softmax_stats_match_oracle(V, T):
    E = _gpu()
    x = W.per_seq_normal(3, (37, V), 2.0, 10, W.TAG_TARGET).reshape(111, V)
    x[5, 17] = x[5].max() + 1.0
    x[6, 3] = x[6, 9] = x[6].max() + 1.0                     # tie: lowest index wins
    m, Z, am, st = oracle.softmax_rows(x, T)
    gm, gz, ga = E.eagle_softmax_stats(_cuda(x), T)
    torch.cuda.synchronize()
    assert np.array_equal(ga.cpu().numpy(), am)
    if T > 0:
        np.testing.assert_allclose(gm.cpu().numpy(), m, rtol=1e-6)
        np.testing.assert_allclose(gz.cpu().numpy(), Z, rtol=1e-5)


@pytest.mark.parametrize("argmax", [True, False])
def test_softmax_stats_full_size_sampled_rows(argmax):
    """B*n = 3840 rows of V = 128256 on the GPU, with and without the argmax (the
    statistics-only variant is the one a T > 0 walk needs); 64 sampled rows checked by
    the oracle."""
    E = _gpu()
    B, n, V = 64, 60, 128256
    x = W.per_seq_normal(B, (n, V), 2.0, 11, W.TAG_TARGET)
    gm, gz, ga = E.eagle_softmax_stats(_cuda(x), 1.0, argmax=argmax)
    torch.cuda.synchronize()
    rows = W.rng(11, 1).choice(B * n, size=64, replace=False)
    flat = x.reshape(B * n, V)[rows]
    m, Z, am, _ = oracle.softmax_rows(flat, 1.0)
    np.testing.assert_allclose(gm.reshape(-1).cpu().numpy()[rows], m, rtol=1e-6)
    np.testing.assert_allclose(gz.reshape(-1).cpu().numpy()[rows], Z, rtol=1e-5)
    if argmax:
        assert np.array_equal(ga.reshape(-1).cpu().numpy()[rows], am)
    else:
        assert ga is None


# ---------------------------------------------------------------- draft vocabulary (d2t)
def _d2t_case(cfg, B, seed, V, Vd, sigma=None):
    d2t, ids = W.d2t_table(V, Vd, seed)
    trow, drows = W.tree_draft_rows_d2t(cfg, seed, ids, B=B, V=V, sigma=sigma)
    tree = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n, d2t=d2t)
    tgt = W.assemble_target(trow, tree["draft_row"], tree["cand"], cfg.target_std, seed)
    return tgt, drows, tree, d2t


def test_d2t_inverse_table_and_bad_tables():
    E = _gpu()
    V, Vd = 1000, 250
    d2t, ids = W.d2t_table(V, Vd, 3)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2d = E.eagle_d2t_inverse(_cuda(d2t), V, dev_status=st).cpu().numpy()
    torch.cuda.synchronize()
    ref = np.full(V, -1, np.int32)
    ref[ids] = np.arange(Vd)
    assert int(st.item()) == 0 and np.array_equal(t2d, ref)
    bad = d2t.copy()
    bad[7] = ids[3] - 7                      # draft id 7 onto draft id 3's target id
    st.zero_()
    E.eagle_d2t_inverse(_cuda(bad), V, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 2                 # EAGLE_DEV_BAD_TOKEN
    out = d2t.copy()
    out[-1] = V - (Vd - 1)                    # last draft id -> target id V
    st.zero_()
    E.eagle_d2t_inverse(_cuda(out), V, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 2


@pytest.mark.parametrize("V,Vd,T", [(128256, 32000, 1.0), (128256, 32000, 0.0), (1000, 252, 1.0),
                                    (1003, 257, 1.0)])
def test_d2t_trees_match_oracle(V, Vd, T):
    """Draft rows over a draft vocabulary of Vd ids mapped to target ids (EAGLE-3's
    32000 of 128256, and ragged small sizes that take the scalar path), 48-node depth-6
    trees built from those rows, B = 8."""
    E = _gpu()
    cfg = W.CONFIGS["sweep_70b"]
    tgt, drows, tree, d2t = _d2t_case(cfg, 8, seed=17, V=V, Vd=Vd)
    ref = oracle.verify_accept_d2t(tgt, drows, d2t, tree["tokens"], tree["parent"], cfg.depth, T,
                                   seed=21, draft_row=tree["draft_row"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2d = E.eagle_d2t_inverse(_cuda(d2t), V, dev_status=st)
    rs = torch.full((2, 8, cfg.n, 2), float("nan"), device="cuda")
    acc, path, emit = E.eagle_verify_accept(
        _cuda(tgt), _cuda(drows), _cuda(tree["tokens"]), _cuda(tree["parent"]), cfg.depth, T, 21,
        draft_row=_cuda(tree["draft_row"]), row_stats=rs, dev_status=st, t2d=t2d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and (ref["status"] == 0).all()
    dec, ties = compare_walks(ref, acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(),
                              exact=(T == 0.0),
                              rows=(tgt, oracle.d2t_scatter(drows, d2t, V), tree["draft_row"], T))
    assert_tie_budget(dec, ties)
    # a random quarter of the target ids leaves most of q's mass outside the draft
    # vocabulary, so acceptance is low; some drafts are still accepted
    assert (ref["accept_len"] > 0).any()
    if T > 0:
        # draft statistics of the visited rows are over the Vd draft ids
        r = rs.cpu().numpy()
        rows = tree["draft_row"]
        seen = ~np.isnan(r[1, :, :, 0])
        assert seen.any()
        m, Z, _, _ = oracle.softmax_rows(drows, T)
        b_i, n_i = np.nonzero(seen)
        np.testing.assert_allclose(r[1, b_i, n_i, 1], Z[b_i, rows[b_i, n_i]], rtol=1e-5)


def test_target_logits_in_pinned_host_memory_give_the_same_walk():
    """target_logits may live in page-locked host memory, read in place by the walk:
    the outputs equal those of the same call on a device copy, bit for bit."""
    E = _gpu()
    cfg = W.CONFIGS["sweep_70b"]
    tgt, drows, tree = _tree_case(cfg, 8, seed=41, V=32000)
    args = (_cuda(drows), _cuda(tree["tokens"]), _cuda(tree["parent"]), cfg.depth, 1.0, 17)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev_out = E.eagle_verify_accept(_cuda(tgt), *args, draft_row=_cuda(tree["draft_row"]),
                                    dev_status=st)
    host = torch.from_numpy(np.ascontiguousarray(tgt)).pin_memory()
    host_out = E.eagle_verify_accept(host, *args, draft_row=_cuda(tree["draft_row"]), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for a, b in zip(dev_out, host_out):
        assert torch.equal(a, b)


# ---------------------------------------------------------------- top-k / top-p filtering
@pytest.mark.parametrize("V,top_k,top_p,quant", [(32000, 50, 0.0, 0.0), (32000, 0, 0.9, 0.0),
                                                 (32000, 20, 0.8, 0.0), (1003, 7, 0.0, 0.5),
                                                 (1003, 0, 0.7, 0.5), (1003, 30, 0.95, 0.25),
                                                 (32000, 100, 0.0, 2.0), (32000, 0, 0.9, 2.0),
                                                 (32000, 3000, 0.99, 0.0)])
def test_filtered_trees_match_oracle(V, top_k, top_p, quant):
    """Top-k / top-p filtered walk on 48-node depth-6 trees, B = 8, against
    oracle.verify_accept_filtered.  quant > 0 rounds every logit to a multiple of quant,
    so cuts fall inside runs of equal logits (the lower token is kept first); at quant 2
    the runs hold thousands of tokens, more than the sorted path takes, so the radix
    select decides.  The
    visited rows' filtered sums (row_stats) are checked to 1e-5."""
    E = _gpu()
    cfg = W.CONFIGS["sweep_70b"]
    tgt, drows, tree = _tree_case(cfg, 8, seed=53, V=V)
    if quant:
        tgt = (np.round(tgt / quant) * quant).astype(np.float32)
        drows = (np.round(drows / quant) * quant).astype(np.float32)
    ref = oracle.verify_accept_filtered(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0,
                                        seed=29, top_k=top_k, top_p=top_p,
                                        draft_row=tree["draft_row"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs = torch.full((2, 8, cfg.n, 2), float("nan"), device="cuda")
    acc, path, emit = E.eagle_verify_accept(
        _cuda(tgt), _cuda(drows), _cuda(tree["tokens"]), _cuda(tree["parent"]), cfg.depth, 1.0, 29,
        draft_row=_cuda(tree["draft_row"]), row_stats=rs, dev_status=st, top_k=top_k, top_p=top_p)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and (ref["status"] == 0).all()
    ft = oracle.filter_logits(tgt, 1.0, top_k, top_p)
    fd = oracle.filter_logits(drows, 1.0, top_k, top_p)
    dec, ties = compare_walks(ref, acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(),
                              rows=(ft, fd, tree["draft_row"], 1.0))
    assert_tie_budget(dec, ties)
    r = rs.cpu().numpy()
    m, Z, _, _ = oracle.softmax_rows(ft, 1.0)
    seen = ~np.isnan(r[0, :, :, 0])
    assert seen.sum() >= 8
    np.testing.assert_allclose(r[0][..., 1][seen], Z[seen], rtol=1e-5)
    _, Zd, _, _ = oracle.softmax_rows(fd, 1.0)
    rows = tree["draft_row"]
    seen = ~np.isnan(r[1, :, :, 0])
    b_i, n_i = np.nonzero(seen)
    np.testing.assert_allclose(r[1, b_i, n_i, 1], Zd[b_i, rows[b_i, n_i]], rtol=1e-5)


def test_filtered_walk_with_fast_and_fallback_rows_in_one_call():
    """Each visited node's two rows take different paths of the cluster filter: the
    target rows are smooth (the cut found from the merged near-bin histogram and the
    gathered candidates), the draft rows quantised to multiples of 2 (thousands of equal
    logits at the cut: the one-CTA radix select).  Sequence 0's target rows are all
    equal, so every token ties and the cut is by index alone.  Against
    oracle.verify_accept_filtered; the visited rows' filtered sums to 1e-5."""
    E = _gpu()
    cfg = W.CONFIGS["sweep_70b"]
    B, top_k, top_p = 8, 50, 0.9
    tgt, drows, tree = _tree_case(cfg, B, seed=57, V=32000)
    drows = (np.round(drows / 2.0) * 2.0).astype(np.float32)
    tgt[0] = 1.5
    ref = oracle.verify_accept_filtered(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0,
                                        seed=37, top_k=top_k, top_p=top_p,
                                        draft_row=tree["draft_row"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs = torch.full((2, B, cfg.n, 2), float("nan"), device="cuda")
    acc, path, emit = E.eagle_verify_accept(
        _cuda(tgt), _cuda(drows), _cuda(tree["tokens"]), _cuda(tree["parent"]), cfg.depth, 1.0, 37,
        draft_row=_cuda(tree["draft_row"]), row_stats=rs, dev_status=st, top_k=top_k, top_p=top_p)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and (ref["status"] == 0).all()
    ft = oracle.filter_logits(tgt, 1.0, top_k, top_p)
    fd = oracle.filter_logits(drows, 1.0, top_k, top_p)
    dec, ties = compare_walks(ref, acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(),
                              rows=(ft, fd, tree["draft_row"], 1.0))
    assert_tie_budget(dec, ties)
    r = rs.cpu().numpy()
    _, Z, _, _ = oracle.softmax_rows(ft, 1.0)
    seen = ~np.isnan(r[0, :, :, 0])
    assert seen[0].any() and seen.sum() >= 8
    np.testing.assert_allclose(r[0][..., 1][seen], Z[seen], rtol=1e-5)
    _, Zd, _, _ = oracle.softmax_rows(fd, 1.0)
    rows = tree["draft_row"]
    seen = ~np.isnan(r[1, :, :, 0])
    b_i, n_i = np.nonzero(seen)
    np.testing.assert_allclose(r[1, b_i, n_i, 1], Zd[b_i, rows[b_i, n_i]], rtol=1e-5)


@pytest.mark.parametrize("B,quant", [(100, 0.0), (160, 0.5), (320, 0.0)])
def test_filtered_walk_at_every_cluster_size(B, quant):
    """The walk's cluster shrinks as B grows (8 CTAs per sequence up to B = 76, then 4,
    2 and, above B = 304, one); the filtered walk splits each visited row's filter over
    the cluster's vocabulary slices (rows it leaves over go to rank 0 for the target and
    rank 1 for the draft, or both to rank 0 in a one-CTA cluster).  Small trees
    (16 nodes, depth 4, 4 children per level) over V = 1003, top-k 12 and top-p 0.8,
    against oracle.verify_accept_filtered."""
    import dataclasses
    E = _gpu()
    cfg = dataclasses.replace(W.CONFIGS["sweep_70b"], n=16, depth=4, top_k=4)
    tgt, drows, tree = _tree_case(cfg, B, seed=61, V=1003)
    if quant:
        tgt = (np.round(tgt / quant) * quant).astype(np.float32)
        drows = (np.round(drows / quant) * quant).astype(np.float32)
    ref = oracle.verify_accept_filtered(tgt, drows, tree["tokens"], tree["parent"], cfg.depth, 1.0,
                                        seed=31, top_k=12, top_p=0.8, draft_row=tree["draft_row"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, path, emit = E.eagle_verify_accept(
        _cuda(tgt), _cuda(drows), _cuda(tree["tokens"]), _cuda(tree["parent"]), cfg.depth, 1.0, 31,
        draft_row=_cuda(tree["draft_row"]), dev_status=st, top_k=12, top_p=0.8)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and (ref["status"] == 0).all()
    rows = (oracle.filter_logits(tgt, 1.0, 12, 0.8), oracle.filter_logits(drows, 1.0, 12, 0.8),
            tree["draft_row"], 1.0)
    dec, ties = compare_walks(ref, acc.cpu().numpy(), path.cpu().numpy(), emit.cpu().numpy(),
                              rows=rows)
    assert_tie_budget(dec, ties)
