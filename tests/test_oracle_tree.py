"""Pins for the oracle's EAGLE-2 expansion / rerank and for KV compaction.

Expansion and rerank: hand-worked examples from the Guide's EAGLE-2 section
(tests/golden/eagle2_rerank_hand.json), a brute-force re-selection, and the
invariants the method fixes (ancestor-closed, topological, exactly n nodes,
depth <= D, kept values >= dropped values).
Compaction: the Lesson's two-sequence rollback exercise
(tests/golden/kv_rollback_two_sequences.json) and overlapping moves.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _hand_cases():
    return json.load(open(os.path.join(GOLD, "eagle2_rerank_hand.json")))["cases"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_eagle2_hand_worked_examples(case):
    t = oracle.Eagle2Tree(case["top_k"], case["depth"])
    for lvl, spec in enumerate(case["levels"]):
        fr = t.expand(np.array(spec["tok"]), np.array(spec["conf"], np.float32))
        assert fr == case["frontiers"][lvl]
    out = t.rerank(case["n_out"])
    for key, val in case["expect"].items():
        assert list(out[key]) == val, key


def _check_tree_invariants(out, trees, n_out, depth):
    B = out["parent"].shape[0]
    for b in range(B):
        par = out["parent"][b]
        cand = out["cand"][b]
        tr = trees[b]
        assert len(par) == n_out and par[0] == -1
        assert all(0 <= par[i] < i for i in range(1, n_out))            # topological
        assert len(set(cand.tolist())) == n_out
        for i in range(1, n_out):                                       # parent map is right
            assert cand[par[i]] == tr.parent[int(cand[i])]
        dep = [tr.depth[int(c)] for c in cand]
        assert max(dep) <= depth
        assert all(dep[i] >= dep[i - 1] for i in range(1, n_out))       # depth ascending
        kept = set(int(c) for c in cand[1:])
        dropped = [c for c in tr.value if c != 0 and c not in kept]
        if dropped:
            assert min(float(tr.value[c]) for c in kept) >= max(float(tr.value[c]) for c in dropped)
        for i in range(1, n_out):                                       # value = parent value * conf
            c = int(cand[i])
            assert tr.value[c] <= tr.value[tr.parent[c]]


def test_eagle2_from_synthetic_logits_invariants():
    cfg = W.CONFIGS["eagle2_b1"]
    B, V = 3, 500
    trow, drows = W.tree_draft_rows(cfg, seed=1, B=B, V=V)
    out = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    _check_tree_invariants(out, out["trees"], cfg.n, cfg.depth)
    # draft rows: every node with children was expanded and owns a row
    for b in range(B):
        par = out["parent"][b]
        for i in set(par[1:].tolist()):
            assert out["draft_row"][b, i] >= 0


def test_eagle2_frontier_is_brute_force_top_k():
    cfg = W.CONFIGS["eagle3_b64"]
    trow, drows = W.tree_draft_rows(cfg, seed=2, B=2, V=300)
    out = oracle.eagle2_from_logits(drows, cfg.top_k, cfg.depth, cfg.n)
    for tr in out["trees"]:
        k = tr.k
        for lvl in range(2, tr.D + 1):
            base = 1 + k + (lvl - 2) * k * k
            ids = list(range(base, base + k * k))
            vals = np.array([float(tr.value[c]) for c in ids])
            # brute force: a candidate is in the frontier iff fewer than k others beat it
            for c, v in zip(ids, vals):
                beats = sum(1 for c2, v2 in zip(ids, vals) if v2 > v or (v2 == v and c2 < c))
                assert (c in tr.frontiers[lvl - 1]) == (beats < k)


def test_eagle2_value_is_float32_product_of_confidences():
    tr = oracle.Eagle2Tree(3, 3)
    g = W.rng(4, 4)
    tr.expand(np.array([[1, 2, 3]]), np.sort(g.random((1, 3)).astype(np.float32))[:, ::-1])
    for _ in range(2):
        tr.expand(g.integers(0, 9, (3, 3)), np.sort(g.random((3, 3)).astype(np.float32))[:, ::-1])
    for c, v in tr.value.items():
        if c == 0:
            continue
        chain, x = [], c
        while x != 0:
            chain.append(x)
            x = tr.parent[x]
        assert tr.depth[c] == len(chain)
        assert v.dtype == np.float32


def test_kv_rollback_two_sequences_exercise():
    spec = json.load(open(os.path.join(GOLD, "kv_rollback_two_sequences.json")))
    nl, B, H, d = 2, 2, 2, 8
    Lmax = 20
    k = W.rng(9, 0).integers(0, 2**16, size=(nl, B, H, Lmax, d)).astype(np.uint16)
    v = k[::-1].copy()
    kv_len = np.array(spec["kv_len_before"], np.int32)
    k0, v0 = k.copy(), v.copy()
    D = spec["n_drafts"]
    st = oracle.kv_compact(k, v, kv_len, np.array(spec["path"], np.int32),
                           np.array(spec["accept_len"], np.int32), D)
    assert st == 0
    assert list(kv_len) == spec["kv_len_after"]
    # chain paths move nothing
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


def test_kv_compact_overlapping_paths_and_untouched_rows():
    nl, B, H, d, Lmax, D = 3, 3, 2, 16, 24, 4
    base = W.rng(1, 1).integers(0, 2**16, size=(nl, B, H, Lmax, d)).astype(np.uint16)
    k, v = base.copy(), base[:, ::-1].copy()
    k0, v0 = k.copy(), v.copy()
    kv_len = np.array([4, 0, 9], np.int32)
    path = np.array([[0, 2, 7, -1, -1],       # row 2 is a source (t=1) and a destination (t=2)
                     [0, 1, 3, 4, 9],
                     [0, -1, -1, -1, -1]], np.int32)
    acc = np.array([2, 4, 0], np.int32)
    st = oracle.kv_compact(k, v, kv_len, path, acc, D)
    assert st == 0 and list(kv_len) == [7, 5, 10]
    for C, C0 in ((k, k0), (v, v0)):
        exp = C0.copy()
        for b, (L, a) in enumerate([(4, 2), (0, 4), (9, 0)]):
            for t in range(a + 1):                  # row L + path[t] of the ORIGINAL cache
                exp[:, b, :, L + t, :] = C0[:, b, :, L + int(path[b, t]), :]
        assert np.array_equal(C, exp)


def test_kv_compact_skips_failed_sequences_and_checks_capacity():
    nl, B, H, d, Lmax, D = 1, 2, 1, 4, 8, 3
    k = np.arange(nl * B * H * Lmax * d, dtype=np.uint16).reshape(nl, B, H, Lmax, d)
    v = k.copy()
    kv_len = np.array([2, 6], np.int32)
    path = np.array([[0, 1, -1, -1], [0, 3, -1, -1]], np.int32)
    st = oracle.kv_compact(k, v, kv_len, path, np.array([-1, 1], np.int32), D)
    assert st == oracle.ORC_CAPACITY and list(kv_len) == [2, 6]


def test_eagle2_with_d2t_maps_tokens_and_keeps_the_tree():
    """A draft vocabulary: the tree (parents, values, draft rows) is the one the draft
    ids give, and each node's token is its draft id's target id d + d2t[d]."""
    B, k, D, n_out, Vd, V = 3, 4, 3, 10, 40, 100
    R = oracle.draft_rows(k, D)
    g = W.rng(3, 46)
    logits = g.normal(0, 2, size=(B, R, Vd)).astype(np.float32)
    ids = np.sort(g.choice(V, size=Vd, replace=False))
    d2t = (ids - np.arange(Vd)).astype(np.int32)
    plain = oracle.eagle2_from_logits(logits, k, D, n_out)
    mapped = oracle.eagle2_from_logits(logits, k, D, n_out, d2t=d2t)
    for key in ("parent", "draft_row", "cand", "value"):
        assert np.array_equal(plain[key], mapped[key])
    assert (mapped["tokens"][:, 0] == -1).all()
    assert np.array_equal(mapped["tokens"][:, 1:], ids[plain["tokens"][:, 1:]])


# ------------------------------------------------------------------ static trees
def test_static_tree_hand_worked_example():
    """Choices (0), (1), (0,0), (0,1), (1,0), (0,0,0), worked out by hand: nodes in
    (length, lexicographic) order after the root."""
    t = oracle.static_tree_from_choices([(1, 0), (0,), (0, 0, 0), (1,), (0, 1), (0, 0)])
    #            root (0)  (1)  (0,0) (0,1) (1,0) (0,0,0)
    assert t["parent"].tolist() == [-1, 0, 0, 1, 1, 2, 3]
    assert t["rank"].tolist() == [-1, 0, 1, 0, 1, 0, 0]
    assert t["depth"].tolist() == [0, 1, 1, 2, 2, 2, 3]
    # internal nodes: root, (0), (1), (0,0) -> rows 0..3
    assert t["draft_row"].tolist() == [0, 1, 2, 3, -1, -1, -1]


def test_static_tree_round_trip_and_errors():
    g = W.rng(8, 47)
    # a random prefix-closed set of choices: grow from the root
    choices = set()
    frontier = [()]
    while frontier and len(choices) < 40:
        c = frontier.pop(0)
        for r in range(int(g.integers(0, 4))):
            choices.add(c + (r,))
            frontier.append(c + (r,))
    choices = sorted(choices, key=lambda c: g.random())           # any input order
    t = oracle.static_tree_from_choices(choices)
    par, rank = t["parent"], t["rank"]
    assert all(0 <= par[i] < i for i in range(1, len(par)))
    paths = set()
    for i in range(1, len(par)):
        p, v = [], i
        while v > 0:
            p.append(int(rank[v]))
            v = par[v]
        paths.add(tuple(reversed(p)))
        assert len(p) == t["depth"][i]
    assert paths == set(choices)
    kids = set(par[1:].tolist())
    assert [i for i in range(len(par)) if t["draft_row"][i] >= 0] == sorted(kids)
    for bad in ([(0,), (0,)], [(1, 0)], [(0,), (-1,)], [()]):
        with pytest.raises(ValueError):
            oracle.static_tree_from_choices(bad)


def test_static_tree_tokens_are_ranked_tokens_of_the_parent_row():
    t = oracle.static_tree_from_choices([(0,), (1,), (2,), (0, 0), (0, 1), (1, 0), (0, 0, 0)])
    R = int(t["draft_row"].max()) + 1
    B, V = 3, 50
    x = W.rng(9, 48).normal(0, 1, size=(B, R, V)).astype(np.float32)
    x[1, 0, 7] = x[1, 0, 3] = x[1, 0].max() + 1        # a tie at the top: lower token first
    tok = oracle.static_tree_tokens(x, t)
    for b in range(B):
        assert tok[b, 0] == -1
        for i in range(1, len(t["parent"])):
            row = x[b, t["draft_row"][t["parent"][i]]].astype(np.float64)
            order = sorted(range(V), key=lambda c: (-row[c], c))
            assert tok[b, i] == order[t["rank"][i]]
    assert tok[1, 1] == 3 and tok[1, 2] == 7
