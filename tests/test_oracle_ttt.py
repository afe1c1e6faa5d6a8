"""Pins for the oracle's training-time-test attention (TTT page, section
"训练时的 attention mask 为什么要特殊处理"): round 0 is causal attention; a simulated
token of round r at position i sees exactly its ancestors in the forest where the
original token i follows token i - 1 and the round-r' token at i follows the round
r' - 1 token at i.

round 0                -> torch scaled_dot_product_attention with is_causal (float64);
any round              -> torch SDPA over every (round, position) key with a boolean
                          mask built from that forest's ancestor closure;
any round, position i  -> the (separately pinned) tree attention with the original
                          rows 0..i-1 as the committed cache and a chain tree of
                          r + 1 nodes (original token i, then rounds 1..r at i);
position 0, round 0    -> its own value row.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _sdpa_ancestors(q, k, v, r, scale):
    """SDPA over all R1 * S keys; query (round r, position i) may see key (r', j) iff
    that token is (r, i) or one of its ancestors, found by following parent links."""
    B, S, Hq, d = q.shape
    Hkv, R1 = k.shape[1], k.shape[2]
    G = Hq // Hkv

    def parent(tok):
        rr, i = tok
        if rr > 0:
            return (rr - 1, i)
        return (0, i - 1) if i > 0 else None

    mask = torch.zeros(S, R1 * S, dtype=torch.bool)
    for i in range(S):
        tok = (r, i)
        while tok is not None:
            mask[i, tok[0] * S + tok[1]] = True
            tok = parent(tok)
    out = torch.zeros(B, S, Hq, d, dtype=torch.float64)
    for b in range(B):
        for h in range(Hq):
            kk = k[b, h // G].double().reshape(R1 * S, d)[None]
            vv = v[b, h // G].double().reshape(R1 * S, d)[None]
            out[b, :, h] = torch.nn.functional.scaled_dot_product_attention(
                q[b, :, h].double()[None], kk, vv, attn_mask=mask[None], scale=scale)[0]
    return out.numpy()


def test_round_zero_is_causal_attention():
    B, S, Hq, Hkv, d, R1 = 2, 11, 4, 2, 16, 3
    q, k, v = W.ttt_inputs(B, S, Hq, Hkv, d, R1, seed=1)
    got = oracle.ttt_attn(q, k, v, 0, 0.3)
    for b in range(B):
        for h in range(Hq):
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[b, :, h].double()[None], k[b, h // 2, 0].double()[None],
                v[b, h // 2, 0].double()[None], is_causal=True, scale=0.3)[0]
            np.testing.assert_allclose(got[b, :, h], ref.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("r", [1, 2, 4])
def test_matches_sdpa_over_the_ancestor_forest(r):
    B, S, Hq, Hkv, d, R1 = 2, 9, 4, 2, 16, 5
    q, k, v = W.ttt_inputs(B, S, Hq, Hkv, d, R1, seed=2)
    scale = d ** -0.5
    got = oracle.ttt_attn(q, k, v, r, scale)
    np.testing.assert_allclose(got, _sdpa_ancestors(q, k, v, r, scale), rtol=1e-12, atol=1e-12)


def test_equals_tree_attention_over_a_chain_per_position():
    B, S, Hq, Hkv, d, R1, r = 1, 7, 2, 1, 32, 4, 3
    q, k, v = W.ttt_inputs(B, S, Hq, Hkv, d, R1, seed=3)
    got = oracle.ttt_attn(q, k, v, r, 0.2)
    n = r + 1
    for i in range(S):
        # cache rows 0..i-1 = original tokens; tree rows i .. i+r = original token i,
        # then the round-1..r tokens at position i
        kc = torch.cat([k[:, :, 0, :i], k[:, :, 0:n, i]], dim=2)
        vc = torch.cat([v[:, :, 0, :i], v[:, :, 0:n, i]], dim=2)
        qq = q[:, i:i + 1].expand(1, n, Hq, d).contiguous()
        ref = oracle.tree_attn(qq, kc, vc, np.array([i], np.int32), W.chain_tree(n)[None], 0.2)
        np.testing.assert_allclose(got[0, i], ref[0, r], rtol=1e-12, atol=1e-13)


def test_first_position_of_round_zero_returns_its_value_row():
    q, k, v = W.ttt_inputs(1, 5, 3, 1, 8, 2, seed=4)
    got = oracle.ttt_attn(q, k, v, 0, 0.5)
    for h in range(3):
        np.testing.assert_array_equal(got[0, 0, h], v[0, 0, 0, 0].double().numpy())


def test_rejects_a_round_outside_the_stored_ones():
    q, k, v = W.ttt_inputs(1, 4, 2, 1, 8, 2, seed=5)
    for r in (-1, 2):
        with pytest.raises(ValueError):
            oracle.ttt_attn(q, k, v, r, 1.0)
