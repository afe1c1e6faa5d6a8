"""Pins for the oracle's numeric kernels against library routines and special cases.

softmax statistics -> scipy logsumexp / torch softmax in float64;
tree attention     -> torch scaled_dot_product_attention (float64, explicit boolean
                      mask); a chain tree is causal attention; a lone root with an
                      empty cache returns its own value row;
LM-head rows       -> numpy float64 matmul;
row top-k          -> numpy stable argsort + float64 softmax.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
import workloads as W


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_stats_match_logsumexp(T):
    x = W.normal((7, 3001), 2.0, 1, 1)
    m, Z, am, st = oracle.softmax_rows(x, T)
    z = x.astype(np.float64) / T
    assert (st == 0).all()
    assert np.array_equal(m, z.max(-1))
    np.testing.assert_allclose(np.log(Z) + m, logsumexp(z, axis=-1), rtol=1e-13)
    ref = torch.softmax(torch.from_numpy(z), -1).numpy()
    prob = np.exp(z - m[:, None]) / Z[:, None]
    np.testing.assert_allclose(prob, ref, rtol=1e-12, atol=1e-300)


def test_softmax_argmax_and_nonfinite_rows():
    x = np.array([[1, 5, 5, 2], [-np.inf, 0, -np.inf, -1], [0, np.nan, 1, 2], [np.inf, 0, 0, 0],
                  [-np.inf] * 4], np.float32)
    m, Z, am, st = oracle.softmax_rows(x, 0.0)
    assert am[0] == 1 and am[1] == 1
    assert list(st) == [0, 0, oracle.ORC_NONFINITE, oracle.ORC_NONFINITE, oracle.ORC_NONFINITE]
    m1, Z1, _, _ = oracle.softmax_rows(x[1:2], 1.0)
    np.testing.assert_allclose(np.log(Z1[0]) + m1[0], logsumexp([0.0, -1.0]), rtol=1e-14)


def _attn_torch(q, k, v, kv_len, parent, scale):
    """Reference: torch SDPA in float64 with an explicit boolean mask."""
    B, n, Hq, d = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = torch.zeros(B, n, Hq, d, dtype=torch.float64)
    for b in range(B):
        L = int(kv_len[b])
        anc, _ = oracle.tree_check(parent[b])
        mask = torch.zeros(n, L + n, dtype=torch.bool)
        mask[:, :L] = True
        for i in range(n):
            for j in range(n):
                mask[i, L + j] = bool((int(anc[i]) >> j) & 1)
        for h in range(Hq):
            qq = q[b, :, h].double()[None]
            kk = k[b, h // G, :L + n].double()[None]
            vv = v[b, h // G, :L + n].double()[None]
            out[b, :, h] = torch.nn.functional.scaled_dot_product_attention(
                qq, kk, vv, attn_mask=mask[None], scale=scale)[0]
    return out.numpy()


def test_tree_attention_matches_sdpa_with_mask():
    B, n, Hq, Hkv, d = 2, 9, 4, 2, 16
    kv_len = np.array([5, 0], np.int32)
    Lmax = 5 + n + 3
    q, k, v, kv_len = W.attn_inputs(B, n, Hq, Hkv, d, kv_len, Lmax, seed=3)
    parent = np.stack([W.random_tree(n, 4, 3, b) for b in range(B)])
    scale = d ** -0.5
    got = oracle.tree_attn(q, k, v, kv_len, parent, scale)
    ref = _attn_torch(q, k, v, kv_len, parent, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_chain_tree_is_causal_attention():
    B, n, Hq, Hkv, d, L = 1, 7, 2, 1, 32, 6
    q, k, v, kv_len = W.attn_inputs(B, n, Hq, Hkv, d, L, L + n, seed=4)
    got = oracle.tree_attn(q, k, v, kv_len, W.chain_tree(n)[None], 0.2)
    for h in range(Hq):
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[0, :, h].double()[None], k[0, 0].double()[None], v[0, 0].double()[None],
            attn_mask=torch.ones(n, L + n, dtype=torch.bool).tril(L)[None], scale=0.2)[0]
        np.testing.assert_allclose(got[0, :, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_lone_root_with_empty_cache_returns_its_value_row():
    q, k, v, kv_len = W.attn_inputs(1, 1, 3, 1, 8, 0, 4, seed=5)
    got = oracle.tree_attn(q, k, v, kv_len, np.array([[-1]]), 0.5)
    for h in range(3):
        np.testing.assert_array_equal(got[0, 0, h], v[0, 0, 0].double().numpy())


def test_tree_attention_rejects_overflow_and_bad_tree():
    q, k, v, kv_len = W.attn_inputs(1, 3, 2, 1, 8, 4, 6, seed=6)
    with pytest.raises(ValueError):
        oracle.tree_attn(q, k, v, kv_len, np.array([[-1, 0, 1]]), 1.0)   # 4 + 3 > 6
    with pytest.raises(ValueError):
        oracle.tree_attn(q, k, v, np.array([2], np.int32), np.array([[-1, 2, 0]]), 1.0)


def test_lmhead_rows_match_numpy_matmul():
    h = W.to_bf16(W.normal((11, 257), 1.0, 1, 2))
    w = W.to_bf16(W.normal((301, 257), 0.02, 1, 3))
    rows = np.array([0, 5, 10], np.int32)
    got = oracle.lmhead_rows(h, w, rows)
    ref = h.double().numpy()[rows] @ w.double().numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_row_topk_matches_stable_sort_and_softmax():
    x = W.normal((5, 2000), 1.3, 2, 2)
    x[0, 100] = x[0, 7] = x[0].max() + 1          # tie at the top: lower token first
    x[1, :] = 0.0                                 # all tied
    tok, conf, st = oracle.row_topk(x, 10)
    for r in range(5):
        order = np.argsort(-x[r].astype(np.float64), kind="stable")[:10]
        assert list(tok[r]) == list(order)
        z = x[r].astype(np.float64)
        pr = np.exp(z - logsumexp(z))
        np.testing.assert_allclose(conf[r], pr[order], rtol=1e-12)
    assert list(tok[0, :2]) == [7, 100] and list(tok[1]) == list(range(10))
