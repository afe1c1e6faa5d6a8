"""Pins for the oracle's verify-and-accept walk.

Each test checks the oracle against something the pages or mathematics fix:
  * the Lesson's closed form E[accepted] = (1 - a^(N+1)) / (1 - a) on chains
    whose every draft is accepted with probability exactly a
    (Lesson "推测解码与 EAGLE-3", section "什么决定加速");
  * the Leviathan invariant: emitted tokens are distributed as q whatever p is,
    checked by chi-square over 50,000 steps (sections "不变量" and "第 5 步");
  * greedy decoding reduces to the target's argmax chain (Guide "无损性的来源"
    and "一次 eagenerate 调用": temperature 0 means greedy);
  * exact enumeration of every (accepted path, final token) on small V = 8
    trees, including the [2,2,2] tree of the Lesson's exercise 3, against a
    Monte Carlo of the oracle;
  * the rule's edge cases from the Lesson's steps 1 and 2 (p(x) <= 0 accepts;
    a residual that sums to zero falls back to q).
"""
import itertools

import numpy as np
import pytest
from scipy import stats

import oracle
import workloads as W

NEG = np.float32(-np.inf)


def _logits(prob):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(prob, np.float64)).astype(np.float32)


def _softmax(row):
    x = np.asarray(row, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def _chisq_pvalue(counts, probs):
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    keep = probs > 0
    assert counts[~keep].sum() == 0, "a zero-probability outcome was observed"
    exp = probs[keep] * counts.sum()
    chi2 = ((counts[keep] - exp) ** 2 / exp).sum()
    return stats.chi2.sf(chi2, keep.sum() - 1)


# ------------------------------------------------------------------ closed form
@pytest.mark.parametrize("alpha", [0.5, 0.8, 0.9])
def test_chain_expected_accepted_matches_closed_form(alpha):
    """V = 8: p uniform on {0..3}; q = alpha p + (1 - alpha) uniform{4..7}, so
    sum_x min(p, q) = alpha and each iid draft is accepted with probability alpha."""
    N, V, B = 5, 8, 100_000
    p = np.array([0.25] * 4 + [0.0] * 4)
    q = alpha * p + (1 - alpha) * np.array([0.0] * 4 + [0.25] * 4)
    tgt = np.broadcast_to(_logits(q), (B, N + 1, V))
    drf = np.broadcast_to(_logits(p), (B, N + 1, V))
    tok = W.rng(1, 99, int(alpha * 100)).integers(0, 4, size=(B, N + 1), dtype=np.int32)
    tok[:, 0] = -1
    par = np.broadcast_to(W.chain_tree(N + 1), (B, N + 1))
    res = oracle.verify_accept(tgt, drf, tok, par, max_depth=N, T=1.0, seed=12345)
    a = res["accept_len"]
    assert (res["status"] == 0).all()
    emitted = a + 1
    closed = (1 - alpha ** (N + 1)) / (1 - alpha)
    se = emitted.std() / np.sqrt(B)
    assert abs(emitted.mean() - closed) < 4 * se, (emitted.mean(), closed, se)
    # the whole law of accept_len: P(a = j) = alpha^j (1 - alpha), P(a = N) = alpha^N
    law = np.array([alpha ** j * (1 - alpha) for j in range(N)] + [alpha ** N])
    assert _chisq_pvalue(np.bincount(a, minlength=N + 1), law) > 1e-3
    # every emitted draft token is an accepted draft; the final token is a real token
    rows = np.arange(B)
    assert (res["emit"][rows, a] >= 0).all()


# ------------------------------------------------------------------ losslessness
def test_leviathan_chisquare_v8_50000_steps():
    V, B = 8, 50_000
    g = W.rng(5, 1)
    p = g.dirichlet(np.ones(V))
    q = g.dirichlet(np.ones(V))
    tgt = np.broadcast_to(_logits(q), (B, 2, V))
    drf = np.broadcast_to(_logits(p), (B, 2, V))
    tok = np.full((B, 2), -1, np.int32)
    tok[:, 1] = g.choice(V, size=B, p=p)                   # d ~ p
    par = np.broadcast_to(W.chain_tree(2), (B, 2))
    res = oracle.verify_accept(tgt, drf, tok, par, max_depth=1, T=1.0, seed=2024)
    first = res["emit"][:, 0]
    qs = _softmax(_logits(q))
    assert _chisq_pvalue(np.bincount(first, minlength=V), qs) > 1e-3
    # and not distributed as p (the test has power)
    assert _chisq_pvalue(np.bincount(first, minlength=V), _softmax(_logits(p))) < 1e-6


def _chain_row_first_tokens(tgt_row, drf_row, steps, seed, chunk=1000):
    """First emitted token of `steps` independent one-draft chain steps on fixed rows
    (target q, draft p; the draft token d ~ p).  The target row after the draft only
    feeds the bonus token, never the first one, so it is a one-token row here."""
    V = tgt_row.size
    p = _softmax(drf_row)
    g = W.rng(seed, 7)
    after = np.full(V, NEG)
    after[0] = 0.0
    tgt = np.ascontiguousarray(np.broadcast_to(np.stack([tgt_row, after]), (chunk, 2, V)))
    drf = np.broadcast_to(drf_row, (chunk, 2, V))
    par = np.broadcast_to(W.chain_tree(2), (chunk, 2))
    firsts = []
    for c in range(steps // chunk):
        tok = np.full((chunk, 2), -1, np.int32)
        tok[:, 1] = g.choice(V, size=chunk, p=p)
        res = oracle.verify_accept(tgt, drf, tok, par, max_depth=1, T=1.0, seed=seed * 1000 + c)
        firsts.append(res["emit"][:, 0])
    return np.concatenate(firsts)


def _equal_mass_bins(q, nbins):
    order = np.argsort(q)
    cum = np.cumsum(q[order])
    bins = np.empty(q.size, int)
    bins[order] = np.minimum((cum * nbins).astype(int), nbins - 1)
    return bins, np.bincount(bins, weights=q, minlength=nbins)


def test_leviathan_chisquare_chain_config_rows_binned():
    """A chain-configuration row pair (V = 32000, target ~ N(0, 2^2), draft = target +
    N(0, 0.5^2)): over 50,000 steps the first emitted token, binned into 50 bins of
    equal q mass (df = 49), is distributed as q, for each of 3 seeds (p-value > 1e-3, at
    most one of the three below 0.05); binned against p instead, the test rejects."""
    V, steps = 32000, 50_000
    tgt_row, drf_row = W.chain_logits(1, 1, V, sigma=0.5, target_std=2.0, seed=3)
    tgt_row, drf_row = tgt_row[0, 0], drf_row[0, 0]
    q, p = _softmax(tgt_row), _softmax(drf_row)
    bins, qbin = _equal_mass_bins(q, 50)
    pbin = np.bincount(bins, weights=p, minlength=50)
    pvals = []
    for seed in (1, 2, 3):
        first = _chain_row_first_tokens(tgt_row, drf_row, steps, seed)
        counts = np.bincount(bins[first], minlength=50)
        pvals.append(_chisq_pvalue(counts, qbin))
        assert _chisq_pvalue(counts, pbin) < 1e-6          # the test has power
    assert min(pvals) > 1e-3, pvals
    assert sum(pv < 0.05 for pv in pvals) <= 1, pvals


def test_race_sampler_matches_normalised_weights():
    r = np.array([0.5, 0.0, 2.0, 1.0, 0.0, 0.25, 3.0, 1.25])
    draws = np.array([oracle.race_sample(r, seed=77, b=b) for b in range(100_000)])
    assert _chisq_pvalue(np.bincount(draws, minlength=8), r / r.sum()) > 1e-3


# ------------------------------------------------------------------ greedy
def test_greedy_emits_target_argmax_chain():
    V, N, B = 50, 5, 16
    tgt, drf = W.chain_logits(B, N + 1, V, sigma=0.5, target_std=2.0, seed=4)
    amax = tgt.argmax(-1).astype(np.int32)                 # numpy: first maximum
    par = np.broadcast_to(W.chain_tree(N + 1), (B, N + 1))
    for k in range(N + 1):
        tok = np.full((B, N + 1), -1, np.int32)
        tok[:, 1:k + 1] = amax[:, :k]                      # draft i+1 = argmax after node i
        if k < N:
            tok[:, k + 1] = (amax[:, k] + 1) % V           # then a wrong draft
            tok[:, k + 2:] = amax[:, k + 1:N]
        res = oracle.verify_accept(tgt, drf, tok, par, max_depth=N, T=0.0, seed=0)
        assert (res["accept_len"] == k).all()
        assert (res["emit"][:, :k + 1] == amax[:, :k + 1]).all()


def test_greedy_argmax_takes_lowest_index_on_ties():
    V = 6
    row = np.array([0.0, 3.0, 1.0, 3.0, 3.0, -2.0], np.float32)
    tgt = np.broadcast_to(row, (1, 2, V))
    tok = np.array([[-1, 3]], np.int32)                    # a tied but higher index
    res = oracle.verify_accept(tgt, tgt, tok, np.array([[-1, 0]]), max_depth=1, T=0.0, seed=0)
    assert res["accept_len"][0] == 0 and res["emit"][0, 0] == 1


# ------------------------------------------------------------------ edge cases
def test_zero_draft_probability_is_accepted():
    """Lesson step 1: p(x) <= 0 accepts, whatever u is."""
    V = 4
    tgt = np.array([[[0.0, 1.0, 2.0, 3.0]] * 2], np.float32)
    drf = np.array([[[0.0, NEG, 1.0, 1.0]] * 2], np.float32)
    tok = np.array([[-1, 1]], np.int32)
    u = np.array([[0.0, 0.999999]])
    res = oracle.verify_accept(tgt, drf, tok, np.array([[-1, 0]]), max_depth=1, T=1.0, seed=0,
                               u_override=u)
    assert res["accept_len"][0] == 1 and res["emit"][0, 0] == 1


def test_zero_residual_falls_back_to_q():
    """Lesson step 2: the clamped residual summing to zero keeps q.  With q == p a
    rejection can only be forced (u = 1); the final token must then follow q."""
    V, B = 6, 40_000
    row = np.array([0.5, NEG, 1.5, -1.0, 2.0, NEG], np.float32)
    tgt = np.broadcast_to(row, (B, 2, V))
    g = W.rng(8, 8)
    q = _softmax(row)
    tok = np.full((B, 2), -1, np.int32)
    tok[:, 1] = g.choice(V, size=B, p=q)
    u = np.ones((B, 2))
    res = oracle.verify_accept(tgt, tgt, tok, np.broadcast_to([-1, 0], (B, 2)), max_depth=1,
                               T=1.0, seed=31, u_override=u)
    assert (res["accept_len"] == 0).all()
    assert _chisq_pvalue(np.bincount(res["emit"][:, 0], minlength=V), q) > 1e-3


def test_invalid_trees_and_tokens_are_flagged():
    V = 5
    tgt = np.zeros((3, 3, V), np.float32)
    par = np.array([[-1, 0, 2], [0, 0, 1], [-1, 0, 1]], np.int32)   # forward parent, bad root, ok
    tok = np.array([[-1, 1, 2], [-1, 1, 2], [-1, 1, V]], np.int32)  # last: token out of range
    res = oracle.verify_accept(tgt, tgt, tok, par, max_depth=2, T=1.0, seed=0)
    assert list(res["status"]) == [oracle.ORC_BAD_TREE, oracle.ORC_BAD_TREE, oracle.ORC_BAD_TOKEN]
    assert (res["accept_len"] == -1).all()
    nan = tgt.copy()
    nan[0, 0, 2] = np.nan
    res = oracle.verify_accept(nan[:1], tgt[:1], tok[2:] % V, par[2:], max_depth=2, T=1.0, seed=0)
    assert res["status"][0] == oracle.ORC_NONFINITE


# ------------------------------------------------------------------ exact trees
def _children(parent, v):
    return [c for c in range(len(parent)) if parent[c] == v]


def _residual(qc, p):
    r = np.maximum(0.0, qc - p)
    s = r.sum()
    return qc.copy() if s == 0 else r / s


def exact_outcomes(q_rows, p_rows, tokens, parent):
    """Probability of every (accepted path, final token) of one tree walk, by
    recursion over the accept/reject events (double precision)."""
    out = {}

    def visit(v, path, prob):
        qc = q_rows[v].copy()
        for c in _children(parent, v):
            x = tokens[c]
            px = p_rows[v][x]
            acc = 1.0 if px <= 0 else min(1.0, qc[x] / px)
            if acc > 0:
                visit(c, path + (c,), prob * acc)
            prob *= 1.0 - acc
            qc = _residual(qc, p_rows[v])
        for y in range(len(qc)):
            if qc[y] > 0:
                out[(path, y)] = out.get((path, y), 0.0) + prob * qc[y]

    visit(0, (0,), 1.0)
    return out


def test_iid_siblings_first_token_is_exactly_q():
    """Multi-round rule with k iid siblings x_i ~ p: the first emitted token is
    distributed exactly as q (exact enumeration over all V^k sibling draws)."""
    V, k = 6, 3
    g = W.rng(2, 2)
    p = g.dirichlet(np.ones(V))
    q = g.dirichlet(np.ones(V) * 0.7)
    parent = np.array([-1] + [0] * k)
    marg = np.zeros(V)
    for xs in itertools.product(range(V), repeat=k):
        w = np.prod([p[x] for x in xs])
        tokens = np.array([-1, *xs])
        outc = exact_outcomes([q] + [q] * k, [p] + [p] * k, tokens, parent)
        for (path, y), pr in outc.items():
            first = tokens[path[1]] if len(path) > 1 else y
            marg[first] += w * pr
    assert np.abs(marg - q).max() < 1e-12


def _monte_carlo_vs_exact(parent, V, seed, B=200_000):
    n = len(parent)
    g = W.rng(seed, 3)
    tgt_rows = g.normal(0, 1.5, size=(n, V)).astype(np.float32)
    drf_rows = (tgt_rows + g.normal(0, 1.0, size=(n, V))).astype(np.float32)
    tokens = np.full(n, -1, np.int32)
    for v in range(n):
        kids = _children(parent, v)
        if kids:
            tokens[kids] = g.choice(V, size=len(kids), replace=False)
    q_rows = [_softmax(r) for r in tgt_rows]
    p_rows = [_softmax(r) for r in drf_rows]
    exact = exact_outcomes(q_rows, p_rows, tokens, parent)
    assert abs(sum(exact.values()) - 1.0) < 1e-12
    D = int(oracle.tree_check(parent)[1].max())
    res = oracle.verify_accept(np.broadcast_to(tgt_rows, (B, n, V)),
                               np.broadcast_to(drf_rows, (B, n, V)),
                               np.broadcast_to(tokens, (B, n)), np.broadcast_to(parent, (B, n)),
                               max_depth=max(D, 1), T=1.0, seed=seed)
    assert (res["status"] == 0).all()
    keys = list(exact)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for b in range(B):
        a = res["accept_len"][b]
        path = tuple(int(x) for x in res["path"][b, :a + 1])
        key = (path, int(res["emit"][b, a]))
        assert key in index, key
        counts[index[key]] += 1
        # the emitted drafts are the tokens of the accepted nodes
        assert all(res["emit"][b, t] == tokens[path[t + 1]] for t in range(a))
    probs = np.array([exact[k] for k in keys])
    # pool cells with small expectation into one so the chi-square is valid
    small = probs * B < 5
    c = np.append(counts[~small], counts[small].sum())
    pr = np.append(probs[~small], probs[small].sum())
    assert _chisq_pvalue(c, pr) > 1e-4


def test_tree_222_exact_enumeration():
    """Lesson exercise 3: a [2, 2, 2] tree (eight candidate paths), V = 8."""
    parent = np.array([-1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6], np.int32)
    _monte_carlo_vs_exact(parent, V=8, seed=222)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_small_trees_exact_enumeration(seed):
    parent = W.random_tree(7, 4, seed)
    _monte_carlo_vs_exact(parent, V=8, seed=seed, B=100_000)


# ------------------------------------------------------------------ draft vocabulary (d2t)
def _d2t_case(V, Vd, seed):
    """A one-to-one draft-to-target table: Vd distinct target ids, d2t[d] = id - d."""
    g = W.rng(seed, 41)
    ids = np.sort(g.choice(V, size=Vd, replace=False))
    return (ids - np.arange(Vd)).astype(np.int32), ids


def test_d2t_scatter_places_draft_probabilities_at_target_ids():
    """p(t) over the target vocabulary is the draft softmax at t = d + d2t[d], 0 elsewhere."""
    V, Vd = 11, 5
    d2t, ids = _d2t_case(V, Vd, 1)
    row = W.rng(1, 42).normal(0, 1, size=(2, 3, Vd)).astype(np.float32)
    full = oracle.d2t_scatter(row, d2t, V)
    for i in range(2):
        for j in range(3):
            pf = _softmax(full[i, j])
            pd = _softmax(row[i, j])
            assert np.allclose(pf[ids], pd, rtol=1e-14, atol=0)
            mask = np.ones(V, bool)
            mask[ids] = False
            assert (pf[mask] == 0).all()


def test_d2t_identity_table_is_the_full_vocabulary_walk():
    B, n, V = 64, 9, 16
    g = W.rng(9, 43)
    parent = W.random_tree(n, 4, 9)
    tgt = g.normal(0, 1.5, size=(B, n, V)).astype(np.float32)
    drf = (tgt + g.normal(0, 1.0, size=(B, n, V))).astype(np.float32)
    tok = np.broadcast_to(g.integers(0, V, size=n, dtype=np.int32), (B, n)).copy()
    tok[:, 0] = -1
    par = np.broadcast_to(parent, (B, n))
    D = int(oracle.tree_check(parent)[1].max())
    a = oracle.verify_accept(tgt, drf, tok, par, max_depth=D, T=1.0, seed=5)
    b = oracle.verify_accept_d2t(tgt, drf, np.zeros(V, np.int32), tok, par, max_depth=D, T=1.0,
                                 seed=5)
    for key in ("accept_len", "path", "emit", "status"):
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("seed", [4, 5])
def test_d2t_tree_walk_exact_enumeration(seed):
    """Draft rows over a draft vocabulary of 5 ids mapped into V = 8 target ids: every
    drafted token is a draft id's target, p is zero on the 3 target ids outside the
    table, and the (accepted path, final token) law is the exact recursion's with p in
    target space (the rule stays lossless: the first emitted token is still ~ q)."""
    V, Vd, B = 8, 5, 100_000
    d2t, ids = _d2t_case(V, Vd, seed)
    parent = W.random_tree(6, 3, seed)
    n = len(parent)
    g = W.rng(seed, 44)
    tgt_rows = g.normal(0, 1.5, size=(n, V)).astype(np.float32)
    drf_rows = g.normal(0, 1.5, size=(n, Vd)).astype(np.float32)
    tokens = np.full(n, -1, np.int32)
    for v in range(n):
        kids = _children(parent, v)
        if kids:
            tokens[kids] = ids[g.choice(Vd, size=len(kids), replace=False)]
    q_rows = [_softmax(r) for r in tgt_rows]
    p_rows = [_softmax(r) for r in oracle.d2t_scatter(drf_rows, d2t, V)]
    exact = exact_outcomes(q_rows, p_rows, tokens, parent)
    assert abs(sum(exact.values()) - 1.0) < 1e-12
    D = int(oracle.tree_check(parent)[1].max())
    res = oracle.verify_accept_d2t(np.broadcast_to(tgt_rows, (B, n, V)),
                                   np.broadcast_to(drf_rows, (B, n, Vd)), d2t,
                                   np.broadcast_to(tokens, (B, n)), np.broadcast_to(parent, (B, n)),
                                   max_depth=max(D, 1), T=1.0, seed=seed)
    assert (res["status"] == 0).all()
    keys = list(exact)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for b in range(B):
        a = res["accept_len"][b]
        key = (tuple(int(x) for x in res["path"][b, :a + 1]), int(res["emit"][b, a]))
        assert key in index, key
        counts[index[key]] += 1
    probs = np.array([exact[k] for k in keys])
    small = probs * B < 5
    c = np.append(counts[~small], counts[small].sum())
    pr = np.append(probs[~small], probs[small].sum())
    assert _chisq_pvalue(c, pr) > 1e-4


def test_d2t_leviathan_chisquare_v8():
    """Losslessness with a draft vocabulary: drafts d ~ p over 5 draft ids, mapped to
    target ids, 50,000 one-draft steps on V = 8; the emitted token is distributed as q
    (including the 3 target ids p never proposes)."""
    V, Vd, B = 8, 5, 50_000
    d2t, ids = _d2t_case(V, Vd, 7)
    g = W.rng(7, 45)
    q = g.dirichlet(np.ones(V))
    pd = g.dirichlet(np.ones(Vd))
    tgt = np.broadcast_to(_logits(q), (B, 2, V))
    drf = np.broadcast_to(_logits(pd), (B, 2, Vd))
    tok = np.full((B, 2), -1, np.int32)
    tok[:, 1] = ids[g.choice(Vd, size=B, p=pd)]
    par = np.broadcast_to(W.chain_tree(2), (B, 2))
    res = oracle.verify_accept_d2t(tgt, drf, d2t, tok, par, max_depth=1, T=1.0, seed=77)
    assert (res["status"] == 0).all()
    first = res["emit"][:, 0]
    assert _chisq_pvalue(np.bincount(first, minlength=V), _softmax(_logits(q))) > 1e-3


# ------------------------------------------------------------------ top-k / top-p filtering
def test_filter_keeps_top_k_then_nucleus_and_renormalises():
    """Hand-checked row: probabilities 0.4, 0.3, 0.2, 0.1 (tokens 2, 0, 3, 1)."""
    p = np.array([0.3, 0.1, 0.4, 0.2])
    row = _logits(p)[None]
    keep = lambda k, tp: np.isfinite(oracle.filter_logits(row, 1.0, k, tp))[0]  # noqa: E731
    assert keep(0, 0.0).tolist() == [True, True, True, True]
    assert keep(2, 0.0).tolist() == [True, False, True, False]          # tokens 2 and 0
    assert keep(0, 0.5).tolist() == [True, False, True, False]          # 0.4 < 0.5 <= 0.7
    assert keep(0, 0.39).tolist() == [False, False, True, False]        # 0.4 reaches 0.39
    assert keep(0, 0.75).tolist() == [True, False, True, True]          # 0.9 >= 0.75
    assert keep(3, 0.95).tolist() == [True, False, True, True]          # top-3 mass 0.9: all 3
    # top-p over what top-k kept: 0.4 / 0.7 = 0.571 < 0.6 <= 1.0
    assert keep(2, 0.6).tolist() == [True, False, True, False]
    assert keep(2, 0.5).tolist() == [False, False, True, False]         # 0.571 >= 0.5
    # ties: lower token first
    tie = np.log(np.array([0.25, 0.25, 0.25, 0.25]))[None].astype(np.float32)
    assert np.isfinite(oracle.filter_logits(tie, 1.0, 2, 0.0))[0].tolist() == [True, True, False,
                                                                               False]
    # temperature enters before the nucleus: at T = 4 the row is flatter
    assert keep(0, 0.5).sum() == 2
    assert np.isfinite(oracle.filter_logits(row, 4.0, 0, 0.5))[0].sum() == 2


def test_filtered_walk_is_lossless_for_the_filtered_target():
    """One-draft chains, drafts from the filtered p: the emitted token is distributed as the
    filtered q (top-k = 5 and top-p = 0.8 on V = 8), 50,000 steps."""
    V, B = 8, 50_000
    g = W.rng(11, 51)
    q = g.dirichlet(np.ones(V))
    p = g.dirichlet(np.ones(V))
    k, tp = 5, 0.8
    qf = _softmax(oracle.filter_logits(_logits(q)[None], 1.0, k, tp)[0])
    pf = _softmax(oracle.filter_logits(_logits(p)[None], 1.0, k, tp)[0])
    tgt = np.broadcast_to(_logits(q), (B, 2, V))
    drf = np.broadcast_to(_logits(p), (B, 2, V))
    tok = np.full((B, 2), -1, np.int32)
    tok[:, 1] = g.choice(V, size=B, p=pf)
    par = np.broadcast_to(W.chain_tree(2), (B, 2))
    res = oracle.verify_accept_filtered(tgt, drf, tok, par, 1, 1.0, 91, top_k=k, top_p=tp)
    assert (res["status"] == 0).all()
    first = res["emit"][:, 0]
    assert _chisq_pvalue(np.bincount(first, minlength=V), qf) > 1e-3
    assert (qf > 0).sum() < V          # the filter removed something
