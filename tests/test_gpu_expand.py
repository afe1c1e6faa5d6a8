"""GPU parity of the draft LM-head GEMM (tcgen05) and of EAGLE-2 expansion / rerank.

GEMM: against the oracle's double-precision rows; tolerance 2e-5 of the row's
largest |logit| (bf16 products are exact in fp32, the only error is fp32
accumulation over K).  Expansion: same float32 logits on both sides; tokens,
parents and draft rows must match exactly unless the oracle's path values show
a near-tie (relative gap < 1e-5) at the divergence.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

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


def _expand_gpu(logits, k, D, n_out, hidden_levels=None, w=None):
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
                        out_tokens=tok, out_parent=par, out_draft_row=row, dev_status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), par.cpu().numpy(), row.cpu().numpy(), int(st.item()), lg


def _compare_trees(ref, tok, par, row):
    mism = 0
    for b in range(tok.shape[0]):
        if (np.array_equal(ref["tokens"][b], tok[b]) and np.array_equal(ref["parent"][b], par[b])
                and np.array_equal(ref["draft_row"][b], row[b])):
            continue
        # a divergence is only allowed where the oracle's values hold a near-tie
        vals = np.array(sorted((float(v) for c, v in ref["trees"][b].value.items() if c), reverse=True))
        gaps = np.abs(np.diff(vals)) / np.maximum(vals[1:], 1e-30)
        assert (gaps < 1e-5).any(), f"sequence {b}: tree mismatch without a near-tie"
        mism += 1
    return mism


@pytest.mark.parametrize("name", ["eagle2_b1", "eagle3_b64", "sweep_70b"])
def test_expansion_from_logits_small_vocab(name):
    cfg = W.CONFIGS[name]
    B, V = 6, 3000
    _, drows = W.tree_draft_rows(cfg, seed=7, B=B, V=V)
    ref = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    tok, par, row, st, _ = _expand_gpu(drows, cfg.top_k, cfg.depth, cfg.n)
    assert st == 0
    assert _compare_trees(ref, tok, par, row) <= 1


def test_expansion_full_size_b64_v128256():
    """64 sequences, depth 8, top-10, V = 128256, rerank to 60 nodes."""
    cfg = W.CONFIGS["expand_b64"]
    _, drows = W.tree_draft_rows(cfg, seed=8)
    ref = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    tok, par, row, st, _ = _expand_gpu(drows, cfg.top_k, cfg.depth, cfg.n)
    assert st == 0
    assert _compare_trees(ref, tok, par, row) <= 1


def test_expansion_fed_by_gemm_matches_expansion_of_its_logits():
    """hidden -> tcgen05 GEMM -> expansion gives the same tree as expanding the very
    logits the GEMM wrote (GPU against GPU; the GEMM itself is checked against the
    oracle above), and the tree is valid.  Small Llama-3-8B-like shape (H = 4096)."""
    B, k, D, n_out, H, V = 4, 10, 4, 30, 4096, 8192
    R = 1 + (D - 1) * k
    w = W.lm_head(V, H, 0.02, 9, block=1024).cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, H, l, 9).cuda() for l in range(1, D + 1)]
    logits = torch.zeros(B, R, V, device="cuda")
    tok, par, row, st, lg = _expand_gpu(logits, k, D, n_out, hidden_levels=hid, w=w)
    assert st == 0
    tok2, par2, row2, st2, _ = _expand_gpu(lg.clone(), k, D, n_out)
    assert st2 == 0
    assert np.array_equal(tok, tok2) and np.array_equal(par, par2) and np.array_equal(row, row2)
    for b in range(B):
        assert par[b, 0] == -1 and all(0 <= par[b, i] < i for i in range(1, n_out))
        assert len(set(zip(par[b, 1:].tolist(), tok[b, 1:].tolist()))) == n_out - 1


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


def test_fused_expansion_matches_unfused_expansion():
    """hidden -> GEMM with per-tile partials -> merge gives the tree of the unfused
    path (GEMM, then one pass over the logits) from the same hidden states, except
    where the two fp32 summation orders leave a near-tie (GPU against GPU; the
    unfused path is checked against the oracle above).  B=8, depth 4, V=32000."""
    E = _E()
    B, k, D, n_out, H, V = 8, 10, 4, 30, 1024, 32000
    R = 1 + (D - 1) * k
    w = W.lm_head(V, H, 0.02, 12, block=1024).cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, H, l, 12).cuda() for l in range(1, D + 1)]
    part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")

    def run(fused):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device="cuda")
        lg = torch.zeros(B, R, V, device="cuda")
        tok = torch.empty(B, n_out, dtype=torch.int32, device="cuda")
        par, row = torch.empty_like(tok), torch.empty_like(tok)
        for lvl in range(1, D + 1):
            E.eagle2_expand(lvl, lvl == D, lg, k, D, n_out, state, hidden=hid[lvl - 1], lm_head_w=w,
                            out_tokens=tok, out_parent=par, out_draft_row=row, dev_status=st,
                            partials=part if fused else None)
        torch.cuda.synchronize()
        return tok.cpu().numpy(), par.cpu().numpy(), row.cpu().numpy(), int(st.item()), lg

    t1, p1, r1, s1, lg1 = run(True)
    t0, p0, r0, s0, lg0 = run(False)
    assert s0 == 0 and s1 == 0
    assert torch.equal(lg0, lg1)                       # the logits rows are written either way
    same = [(np.array_equal(t1[b], t0[b]) and np.array_equal(p1[b], p0[b]) and
             np.array_equal(r1[b], r0[b])) for b in range(B)]
    assert sum(same) >= B - 1


def _expand_tree(E, B, k, D, n_out, V, w, hid, part):
    R = 1 + (D - 1) * k
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device="cuda")
    lg = torch.zeros(B, R, V, device="cuda")
    tok = torch.empty(B, n_out, dtype=torch.int32, device="cuda")
    par, row = torch.empty_like(tok), torch.empty_like(tok)
    for lvl in range(1, D + 1):
        E.eagle2_expand(lvl, lvl == D, lg, k, D, n_out, state, hidden=hid[lvl - 1], lm_head_w=w,
                        out_tokens=tok, out_parent=par, out_draft_row=row, dev_status=st,
                        partials=part)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), par.cpu().numpy(), row.cpu().numpy(), int(st.item())


def test_fused_expansion_tied_logits():
    """LM-head rows repeated with period 500, so every logit of a row occurs 64 times
    in 64 different tiles: the k largest tile maxima all tie, every one of the 64
    tiles holding the row's best value is read back, and the top-k must be the k
    lowest columns of that value, as the one-pass top-k gives.  Within a row the
    children's path values tie exactly, so fused and unfused trees agree token for
    token.  B=8, k=10, depth 3, V=32000."""
    E = _E()
    B, k, D, n_out, H, V = 8, 10, 3, 20, 512, 32000
    base = W.lm_head(500, H, 0.02, 13, block=500)
    w = base.repeat(V // 500, 1).contiguous().cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, H, l, 13).cuda() for l in range(1, D + 1)]
    part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")
    t1, p1, r1, s1 = _expand_tree(E, B, k, D, n_out, V, w, hid, part)
    t0, p0, r0, s0 = _expand_tree(E, B, k, D, n_out, V, w, hid, None)
    assert s0 == 0 and s1 == 0
    for b in range(B):
        # level-1 children: the 10 lowest columns of the root row's best value
        kids = sorted(t1[b, 1:][p1[b, 1:] == 0].tolist())
        assert len(kids) > 0
        assert all(t % 500 == kids[0] % 500 for t in kids)
    assert np.array_equal(t1, t0) and np.array_equal(p1, p0) and np.array_equal(r1, r0)


@pytest.mark.parametrize("fused", [False, True])
def test_expansion_with_d2t_matches_oracle(fused):
    """A draft vocabulary of 8000 ids of a 32000-id target vocabulary: the GPU tree's
    tokens are the mapped target ids, the tree is the oracle's.  Given logits
    (one-pass top-k), or from hidden states through the GEMM (fused top-k; the oracle
    then expands the very logits the GEMM wrote)."""
    E = _E()
    B, k, D, n_out, H, V, Vt = 4, 10, 4, 30, 512, 8000, 32000
    d2t, ids = W.d2t_table(Vt, V, 5)
    R = 1 + (D - 1) * k
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device="cuda")
    tok = torch.empty(B, n_out, dtype=torch.int32, device="cuda")
    par, row = torch.empty_like(tok), torch.empty_like(tok)
    front = torch.empty(B, k, dtype=torch.int32, device="cuda")
    d2t_gpu = torch.from_numpy(d2t).cuda()
    if fused:
        w = W.lm_head(V, H, 0.02, 6, block=1000).cuda()
        hid = [W.hidden_states(B, 1 if l == 1 else k, H, l, 6).cuda() for l in range(1, D + 1)]
        lg = torch.zeros(B, R, V, device="cuda")
        part = torch.empty(E.expand_scratch_size(B, V, k) // 4, device="cuda")
    else:
        cfg = W.CONFIGS["eagle3_b64"]
        _, drows = W.tree_draft_rows(cfg, seed=6, B=B, V=V)
        lg = torch.from_numpy(np.ascontiguousarray(drows[:, :R])).cuda()
    for lvl in range(1, D + 1):
        E.eagle2_expand(lvl, lvl == D, lg, k, D, n_out, state,
                        hidden=hid[lvl - 1] if fused else None, lm_head_w=w if fused else None,
                        out_tokens=tok, out_parent=par, out_draft_row=row, frontier_tokens=front,
                        dev_status=st, partials=part if fused else None, d2t=d2t_gpu)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.eagle2_from_logits(lg.cpu().numpy(), k, D, n_out, d2t=d2t)
    assert _compare_trees(ref, tok.cpu().numpy(), par.cpu().numpy(), row.cpu().numpy()) <= 1
    t = tok.cpu().numpy()[:, 1:]
    assert np.isin(t, ids).all()
    assert np.isin(front.cpu().numpy(), ids).all()
