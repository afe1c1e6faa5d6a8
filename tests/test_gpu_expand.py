"""GPU parity of the draft LM-head GEMM (tcgen05) and of EAGLE-2 expansion / rerank.

GEMM: against the oracle's double-precision rows; tolerance 2e-5 of the row's
largest |logit| (bf16 products are exact in fp32, the only error is fp32
accumulation over K).

Expansion (tests.helpers.check_expansion): every sequence's selection is replayed
by the oracle on the GPU's own confidences and must reproduce parents, float32
path values, frontiers and the reranked tree exactly; per-row top-k tokens equal
the oracle's (on GEMM-computed rows, a swap only where the oracle's fp64 logits
differ by less than the two logits' measured GEMM error); confidences c agree
with the oracle's fp64 ones to 1e-5 relative and path values V with the oracle's
own tree to 1e-5 relative; the oracle's own tree may differ only at a cut whose
two candidates it separates by less than 2e-5 relative.  The oracle's inputs are
the seeded generators' (for GEMM-fed trees it computes the logits itself).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

from tests import helpers as H

pytestmark = pytest.mark.gpu


def _E():
    import eagle_tree_speculative_gb300 as E
    return E


def _gemm_check(M, K, N, rows, seed, **kw):
    E = _E()
    h = W.to_bf16(W.normal((M, K), 1.0, seed, 1))
    w = W.lm_head(N, K, 0.02, seed, block=1024)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = E.eagle_lmhead_gemm(h.cuda(), w.cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.lmhead_rows(h, w, np.asarray(rows, np.int32))
    g = got.cpu().numpy()[rows]
    tol = 2e-5 * np.abs(ref).max(-1, keepdims=True)
    assert (np.abs(g - ref) <= tol).all(), np.abs(g - ref).max()


def test_gemm_small_ragged_all_rows():
    _gemm_check(M=37, K=128, N=300, rows=np.arange(37), seed=1)


def test_gemm_two_m_tiles_and_n_tail():
    _gemm_check(M=200, K=256, N=1000, rows=np.arange(0, 200, 7), seed=2)


def test_gemm_llama3_8b_shape_sampled_rows():
    """M = 640 (64 seqs x 10 frontier rows), K = 4096, N = 128256; 6 rows checked."""
    _gemm_check(M=640, K=4096, N=128256, rows=[0, 127, 128, 333, 511, 639], seed=3)


def test_gemm_row_mapping_into_draft_logit_storage():
    """Rows of one expansion level land at b * R + off + s of the [B, R, V] storage."""
    E = _E()
    B, k_in, R, off, K, N = 5, 3, 9, 4, 128, 520
    h = W.to_bf16(W.normal((B * k_in, K), 1.0, 4, 1))
    w = W.lm_head(N, K, 0.02, 4, block=512)
    out = torch.full((B, R, N), -7.0, device="cuda")
    E.eagle_lmhead_gemm(h.cuda(), w.cuda(), out=out, ldo=N, rows_per_group=k_in, group_stride=R,
                        row_offset=off)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    ref = oracle.lmhead_rows(h, w, np.arange(B * k_in, dtype=np.int32))
    for b in range(B):
        for s in range(k_in):
            np.testing.assert_allclose(o[b, off + s], ref[b * k_in + s], rtol=0,
                                       atol=2e-5 * np.abs(ref).max())
        untouched = [r for r in range(R) if not off <= r < off + k_in]
        assert (o[b, untouched] == -7.0).all()


def _read_cand(E, state, B, k, D):
    c = E.eagle2_tree_candidates(state, B, k, D)
    torch.cuda.synchronize()
    return {name: t.cpu().numpy() for name, t in c.items()}


def _expand_gpu(logits, k, D, n_out, hidden_levels=None, w=None, partials=None, d2t=None):
    """Run every level of one expansion on the GPU; returns (tokens, parent, draft_row,
    status, logits tensor, candidates read back from the tree state)."""
    E = _E()
    B, R, V = logits.shape
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device="cuda")
    tok = torch.empty(B, n_out, dtype=torch.int32, device="cuda")
    par = torch.empty_like(tok)
    row = torch.empty_like(tok)
    lg = logits if isinstance(logits, torch.Tensor) else torch.from_numpy(logits).cuda()
    for lvl in range(1, D + 1):
        hid = None if hidden_levels is None else hidden_levels[lvl - 1]
        E.eagle2_expand(lvl, lvl == D, lg, k, D, n_out, state, hidden=hid, lm_head_w=w,
                        out_tokens=tok, out_parent=par, out_draft_row=row, dev_status=st,
                        partials=partials, d2t=d2t)
    torch.cuda.synchronize()
    cand = _read_cand(E, state, B, k, D)
    return tok.cpu().numpy(), par.cpu().numpy(), row.cpu().numpy(), int(st.item()), lg, cand


def _ref_rows(x, k, d2t=None):
    """The oracle's top-k tokens (target ids) and fp64 confidences of every row."""
    tok, conf, st = oracle.row_topk(x, k)
    assert (st == 0).all()
    if d2t is not None:
        tok = (tok + np.asarray(d2t, np.int64)[tok]).astype(np.int32)
    return tok, conf


def _oracle_gemm_rows(hid, w, seqs, k, D):
    """The oracle's logits (fp64) of every draft row of the sequences `seqs`, computed
    from the level hidden states [B, k_in, H] and W: {b: [R, V]}."""
    R = 1 + (D - 1) * k
    V = w.shape[0]
    out = {b: np.zeros((R, V)) for b in seqs}
    for lvl in range(1, D + 1):
        k_in = 1 if lvl == 1 else k
        h = hid[lvl - 1].reshape(-1, hid[lvl - 1].shape[-1])
        rows = [b * k_in + s for b in seqs for s in range(k_in)]
        got = oracle.lmhead_rows(h, w, np.asarray(rows, np.int32))
        off = oracle.level_row_offset(lvl, k)
        for i, b in enumerate(seqs):
            out[b][off:off + k_in] = got[i * k_in:(i + 1) * k_in]
    return out


def _gemm_tie_check(l64, lg_gpu, seqs):
    """The GEMM's rows against the oracle (2e-5 of the row's largest |logit|), and the
    explanation of a top-k difference: the GPU ranked its own fp32 logits, so two tokens
    may swap only when the oracle separates them by less than the two logits' actual
    errors (plus one float32 rounding of each)."""
    err = {}
    for b in seqs:
        g = lg_gpu[b].astype(np.float64)
        e = np.abs(g - l64[b])
        tol = 2e-5 * np.abs(l64[b]).max(-1, keepdims=True)
        assert (e <= tol).all(), (b, float(e.max()))
        err[b] = e

    def tie_ok(b, r, a, g):
        la, lb = l64[b][r, a], l64[b][r, g]
        ulp = 2.0 ** (np.floor(np.log2(max(abs(la), abs(lb), 1e-30))) - 23)
        return abs(la - lb) <= err[b][r, a] + err[b][r, g] + 2 * ulp

    # each logit's error moves a confidence c_t = exp(l_t - m) / Z by at most
    # |e_t| + max_s |e_s| relative (both fp32 roundings of the oracle's rows included)
    slack = {b: 2.0 * float(err[b].max()) + 2.0 ** -23 for b in seqs}
    return tie_ok, slack


def _own_tree(x32, seqs, k, D, n_out, d2t=None):
    """The oracle's own expansion of the given float32 rows, keyed by sequence."""
    ref = oracle.eagle2_from_logits(np.stack([x32[b] for b in seqs]), k, D, n_out, d2t=d2t)
    return {"trees": {b: ref["trees"][i] for i, b in enumerate(seqs)},
            "tokens": {b: ref["tokens"][i] for i, b in enumerate(seqs)},
            "parent": {b: ref["parent"][i] for i, b in enumerate(seqs)},
            "draft_row": {b: ref["draft_row"][i] for i, b in enumerate(seqs)}}


def _check_given_logits(drows, k, D, n_out, d2t=None, d2t_gpu=None):
    tok, par, row, st, _, cand = _expand_gpu(drows, k, D, n_out, d2t=d2t_gpu)
    assert st == 0
    rt, rc = _ref_rows(drows, k, d2t)
    own = oracle.eagle2_from_logits(drows, k, D, n_out, d2t=d2t)
    stats = H.check_expansion(oracle, cand, (tok, par, row), rt, rc, k, D, n_out, own=own)
    print("expansion parity:", stats)
    assert stats["tie_rows"] == 0
    return stats


@pytest.mark.parametrize("name", ["eagle2_b1", "eagle3_b64", "sweep_70b"])
def test_expansion_from_logits_small_vocab(name):
    """Given logits rows (the one-pass top-k): per-row tokens exact and confidences to
    1e-5, an exact replay of the selection on the GPU's confidences, and values to 1e-5
    of the oracle's own tree, divergences only at the oracle's near-tie cuts."""
    cfg = W.CONFIGS[name]
    _, drows = W.tree_draft_rows(cfg, seed=7, B=6, V=3000)
    _check_given_logits(drows, cfg.top_k, cfg.depth, cfg.n)


def test_expansion_full_size_b64_v128256():
    """64 sequences, depth 8, top-10, V = 128256, rerank to 60 nodes, given logits."""
    cfg = W.CONFIGS["expand_b64"]
    _, drows = W.tree_draft_rows(cfg, seed=8)
    _check_given_logits(drows, cfg.top_k, cfg.depth, cfg.n)


@pytest.fixture(scope="module")
def w_llama3():
    """The Llama-3-8B-shaped draft LM head, W [128256, 4096] bf16 ~ N(0, 0.02^2)."""
    return W.lm_head(128256, 4096, 0.02, 3, block=1024)


def test_bench_fused_expansion_full_size(w_llama3):
    """The expansion exactly as the benchmark step runs it: per level, hidden states ->
    tcgen05 LM-head GEMM with per-tile partials -> top-k merge -> select, then rerank;
    B = 64, H = 4096, V = 128256, depth 8, top-10, 60 nodes.  The oracle computes the
    logits rows of three sampled sequences itself (fp64 from the same hidden states and W)
    and expands them; every sequence's selection is replayed exactly on the GPU's own
    confidences."""
    E = _E()
    B, k, D, n_out, Hd, V = 64, 10, 8, 60, 4096, 128256
    R = 1 + (D - 1) * k
    w = w_llama3.cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, Hd, l, 21) for l in range(1, D + 1)]
    part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")
    lg = torch.empty(B, R, V, device="cuda")
    tok, par, row, st, lg, cand = _expand_gpu(lg, k, D, n_out, hidden_levels=[h.cuda() for h in hid],
                                              w=w, partials=part)
    assert st == 0
    seqs = [0, 29, 63]
    l64 = _oracle_gemm_rows(hid, w_llama3, seqs, k, D)
    gl = {b: lg[b].cpu().numpy() for b in seqs}
    del lg
    tie_ok, slack = _gemm_tie_check(l64, gl, seqs)
    x32 = {b: l64[b].astype(np.float32) for b in seqs}
    rt, rc = {}, {}
    for b in seqs:
        rt[b], rc[b] = _ref_rows(x32[b], k)
    own = _own_tree(x32, seqs, k, D, n_out)
    stats = H.check_expansion(oracle, cand, (tok, par, row), rt, rc, k, D, n_out, own=own,
                              tie_ok=tie_ok, rows_for=seqs, slack=slack)
    print("fused full-size expansion parity:", stats)


def test_fused_expansion_matches_oracle():
    """hidden -> GEMM with per-tile partials -> merge, against the oracle's expansion of
    its own fp64 logits of the same hidden states and W (every sequence and row); the
    unfused path from the same hidden states writes bit-identical logits rows.
    B = 8, depth 4, top-10, H = 1024, V = 32000."""
    E = _E()
    B, k, D, n_out, Hd, V = 8, 10, 4, 30, 1024, 32000
    R = 1 + (D - 1) * k
    w_cpu = W.lm_head(V, Hd, 0.02, 12, block=1024)
    w = w_cpu.cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, Hd, l, 12) for l in range(1, D + 1)]
    part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")
    res = {}
    for fused in (True, False):
        res[fused] = _expand_gpu(torch.zeros(B, R, V, device="cuda"), k, D, n_out,
                                 hidden_levels=[h.cuda() for h in hid], w=w,
                                 partials=part if fused else None)
        assert res[fused][3] == 0
    assert torch.equal(res[True][4], res[False][4])
    seqs = list(range(B))
    l64 = _oracle_gemm_rows(hid, w_cpu, seqs, k, D)
    tie_ok, slack = _gemm_tie_check(l64, res[True][4].cpu().numpy(), seqs)
    x32 = {b: l64[b].astype(np.float32) for b in seqs}
    rt, rc = {}, {}
    for b in seqs:
        rt[b], rc[b] = _ref_rows(x32[b], k)
    own = _own_tree(x32, seqs, k, D, n_out)
    for fused in (True, False):
        tok, par, row, _, _, cand = res[fused]
        stats = H.check_expansion(oracle, cand, (tok, par, row), rt, rc, k, D, n_out, own=own,
                                  tie_ok=tie_ok, slack=slack)
        print("fused" if fused else "unfused", "expansion parity:", stats)


@pytest.mark.parametrize("M,N", [(37, 1000), (200, 2304), (130, 4096 + 77)])
def test_gemm_partials_are_per_tile_statistics(M, N):
    """The epilogue's per-tile partials against the GEMM's own fp32 output: tile max
    bit-exact, sum of 2^((l - max) log2 e) to 1e-5 relative (fp64 reference); ragged
    M and N tails."""
    E = _E()
    K = 256
    h = W.to_bf16(W.normal((M, K), 1.0, 11, M)).cuda()
    w = W.lm_head(N, K, 0.02, 11, block=1024).cuda()
    tiles = (N + 255) // 256
    part = torch.full((M, tiles, 2), float("nan"), device="cuda")
    out = E.eagle_lmhead_gemm(h, w, partials=part)
    torch.cuda.synchronize()
    lg = out.cpu().numpy().astype(np.float64)
    pt = part.cpu().numpy()
    for t in range(tiles):
        blk = lg[:, 256 * t: min(N, 256 * t + 256)]
        mx = blk.max(1)
        assert np.array_equal(pt[:, t, 0].astype(np.float64), mx)
        ssum = np.exp(blk - mx[:, None]).sum(1)
        np.testing.assert_allclose(pt[:, t, 1], ssum, rtol=1e-5)


def test_fused_expansion_tied_logits():
    """LM-head rows repeated with period 500, so every logit of a row occurs 64 times
    in 64 different tiles: the k largest tile maxima all tie, every one of the 64
    tiles holding the row's best value is read back, and the top-k must be the k
    lowest columns of that value (ties to the lower token).  Fused and unfused trees
    are checked against the oracle's expansion of its own fp64 logits.
    B = 8, k = 10, depth 3, V = 32000."""
    E = _E()
    B, k, D, n_out, Hd, V = 8, 10, 3, 20, 512, 32000
    R = 1 + (D - 1) * k
    base = W.lm_head(500, Hd, 0.02, 13, block=500)
    w_cpu = base.repeat(V // 500, 1).contiguous()
    w = w_cpu.cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, Hd, l, 13) for l in range(1, D + 1)]
    part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")
    seqs = list(range(B))
    l64 = _oracle_gemm_rows(hid, w_cpu, seqs, k, D)
    x32 = {b: l64[b].astype(np.float32) for b in seqs}
    rt, rc = {}, {}
    for b in seqs:
        rt[b], rc[b] = _ref_rows(x32[b], k)
        # the oracle's own level-1 children are 10 columns of one repeated logit
        assert len(set((rt[b][0] % 500).tolist())) == 1
    own = _own_tree(x32, seqs, k, D, n_out)
    for fused in (True, False):
        tok, par, row, st, lg, cand = _expand_gpu(
            torch.zeros(B, R, V, device="cuda"), k, D, n_out,
            hidden_levels=[h.cuda() for h in hid], w=w, partials=part if fused else None)
        assert st == 0
        tie_ok, slack = _gemm_tie_check(l64, lg.cpu().numpy(), seqs)
        stats = H.check_expansion(oracle, cand, (tok, par, row), rt, rc, k, D, n_out, own=own,
                                  tie_ok=tie_ok, slack=slack)
        print("fused" if fused else "unfused", "tied-logit expansion parity:", stats)


@pytest.mark.parametrize("fused", [False, True])
def test_expansion_with_d2t_matches_oracle(fused):
    """A draft vocabulary of 8000 ids of a 32000-id target vocabulary: the GPU tree's
    tokens are the mapped target ids, strictly checked against the oracle.  Given logits
    (one-pass top-k), or from hidden states through the GEMM (fused top-k; the oracle
    computes those logits itself from the same hidden states and W)."""
    E = _E()
    B, k, D, n_out, Hd, V, Vt = 4, 10, 4, 30, 512, 8000, 32000
    d2t, ids = W.d2t_table(Vt, V, 5)
    R = 1 + (D - 1) * k
    d2t_gpu = torch.from_numpy(d2t).cuda()
    if not fused:
        cfg = W.CONFIGS["eagle3_b64"]
        _, drows = W.tree_draft_rows(cfg, seed=6, B=B, V=V)
        drows = np.ascontiguousarray(drows[:, :R])
        _check_given_logits(drows, k, D, n_out, d2t=d2t, d2t_gpu=d2t_gpu)
        return
    w_cpu = W.lm_head(V, Hd, 0.02, 6, block=1000)
    hid = [W.hidden_states(B, 1 if l == 1 else k, Hd, l, 6) for l in range(1, D + 1)]
    part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")
    tok, par, row, st, lg, cand = _expand_gpu(
        torch.zeros(B, R, V, device="cuda"), k, D, n_out, hidden_levels=[h.cuda() for h in hid],
        w=w_cpu.cuda(), partials=part, d2t=d2t_gpu)
    assert st == 0
    seqs = list(range(B))
    l64 = _oracle_gemm_rows(hid, w_cpu, seqs, k, D)
    tie_ok, slack = _gemm_tie_check(l64, lg.cpu().numpy(), seqs)
    x32 = {b: l64[b].astype(np.float32) for b in seqs}
    rt, rc = {}, {}
    for b in seqs:
        rt[b], rc[b] = _ref_rows(x32[b], k, d2t)
    own = _own_tree(x32, seqs, k, D, n_out, d2t=d2t)
    stats = H.check_expansion(oracle, cand, (tok, par, row), rt, rc, k, D, n_out, own=own,
                              tie_ok=tie_ok, slack=slack)
    print("d2t fused expansion parity:", stats)
    assert np.isin(tok[:, 1:], ids).all()


def test_frontier_tokens_are_the_frontier():
    """frontier_tokens after each level below the last holds the tokens of the level's
    k best candidates, best first (slot s = draft row 1 + (level-1) k + s)."""
    E = _E()
    cfg = W.CONFIGS["eagle3_b64"]
    B, k, D, n_out, V = 4, cfg.top_k, 4, 30, 3000
    _, drows = W.tree_draft_rows(cfg, seed=14, B=B, V=V)
    R = 1 + (D - 1) * k
    lg = torch.from_numpy(np.ascontiguousarray(drows[:, :R])).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device="cuda")
    tok = torch.empty(B, n_out, dtype=torch.int32, device="cuda")
    par, row = torch.empty_like(tok), torch.empty_like(tok)
    front = torch.empty(B, k, dtype=torch.int32, device="cuda")
    for lvl in range(1, D):
        E.eagle2_expand(lvl, 0, lg, k, D, n_out, state, out_tokens=tok, out_parent=par,
                        out_draft_row=row, frontier_tokens=front, dev_status=st)
        torch.cuda.synchronize()
        cand = _read_cand(E, state, B, k, D)
        f = front.cpu().numpy()
        for b in range(B):
            rows = 1 + (lvl - 1) * k
            ids = [int(np.nonzero((cand["draft_row"][b] == rows + s) &
                                  (cand["depth"][b] == lvl))[0][0]) for s in range(k)]
            assert np.array_equal(f[b], cand["token"][b, ids])
    assert int(st.item()) == 0
