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


@pytest.mark.parametrize("name", ["eagle2_b1", "eagle3_b64"])
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
