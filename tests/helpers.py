"""Comparison helpers shared by the GPU parity tests.

Tolerances (written out here and in each test):
  * integer / index results: bit-exact;
  * temperature 0: bit-exact (decisions compare raw float32 logits on both sides);
  * temperature > 0: accept decisions identical except near-ties, a tested child
    with |u * p(x) - q_cur(x)| < 1e-6 (probabilities from the double-precision
    oracle), or a sampling race whose two best keys (oracle, exact) differ by less
    than the device keys' derived error bound (race_tie_bound); the near-tie count
    must stay below 1e-4 of all decisions (one is tolerated in small runs);
  * probabilities / softmax statistics: 1e-5 relative;
  * bf16 attention output: per (sequence, node, head) row,
    max |O_gpu - O_ref| / max |O_ref| <= 1e-2.
"""
from __future__ import annotations

import math

import numpy as np

NEAR_TIE_ABS = 1e-6

# Error terms of the device's race key w_t / E_t, relative, first order (float32):
EPS_ROUND = 2.0 ** -24     # one correctly rounded float32 operation
EPS_EXP2 = 2.0 ** -22      # exp2f: at most 2 ulp (CUDA math API)
EPS_LOG1P = 2.0 ** -23     # log1pf: at most 1 ulp (CUDA math API); E = -log1pf(-v), v exact
EPS_STAT = 1e-5            # a row's normaliser (sum of exponentials): the statistics tolerance,
                           # checked on every visited row by the row_stats tests


def _softmax64(row, T):
    x = np.asarray(row, np.float64) / T
    m = x[np.isfinite(x)].max()
    e = np.exp(x - m)
    return e / e.sum()


def race_tie_bound(rows, b, v, n_rej, y, y2):
    """Largest relative gap between the exact race keys of tokens y and y2 at node v that
    the device's float32 keys can invert.  The device key of token t is w_t / E_t:
      * E_t = -log1pf(-v_t) with v_t exact: 1 ulp, then one rounding for the division;
      * w_t = 2^((l_t - m) c) / S (bonus, no rejected child): exp2f's 2 ulp, the rounding
        of (l_t - m), of its product with c = log2 e / T and of the float c itself (3
        roundings of the exponent a_t = (m - l_t) c, i.e. 3 ln 2 |a_t| 2^-24 relative),
        and one rounding for the product with 1 / S, which is common to every token;
      * after J rejections of v's children, w_t = max(0, q_t - C p_t) with C the rejection
        recurrence's constant: q_t and p_t each carry the terms above plus their own
        normaliser's error (EPS_STAT, no longer common), and the subtraction amplifies them
        by (q_t + C p_t) / w_t.
    The bound is the sum of the two tokens' errors.  rows = (target [B, n, V], draft
    [B, R, V] over target ids, draft_row [B, n] or None, T)."""
    tgt, drf, draft_row, T = rows
    c = 1.0 / (T * math.log(2.0))
    lq = np.asarray(tgt[b, v], np.float64)
    q = _softmax64(lq, T)
    aq = (lq[np.isfinite(lq)].max() - lq) * c
    eq = EPS_EXP2 + 3 * math.log(2.0) * EPS_ROUND * np.abs(aq) + EPS_ROUND
    if n_rej == 0:
        delta = eq
    else:
        r = int(v if draft_row is None else draft_row[b, v])
        lp = np.asarray(drf[b, r], np.float64)
        p = _softmax64(lp, T)
        with np.errstate(invalid="ignore"):
            ap = np.where(np.isfinite(lp), (lp[np.isfinite(lp)].max() - lp) * c, 0.0)
        ep = EPS_EXP2 + 3 * math.log(2.0) * EPS_ROUND * ap + EPS_ROUND + EPS_STAT
        eq = eq + EPS_STAT
        C, Dj, w = 0.0, 1.0, q
        for j in range(n_rej):
            cn = C + Dj
            wn = np.maximum(0.0, q - cn * p)
            sn = wn.sum()
            if j == n_rej - 1:
                if sn > 0:
                    C, w = cn, wn
            elif sn > 0:
                C, Dj = cn, sn
        with np.errstate(divide="ignore", invalid="ignore"):
            delta = (eq * q + ep * C * p) / w + EPS_ROUND
    delta = delta + EPS_LOG1P + EPS_ROUND
    return float(delta[y] + delta[y2])


def compare_walks(ref, acc, path, emit, exact=False, rows=None):
    """Compare the GPU walk (acc, path, emit numpy arrays) with the oracle's.

    rows = (target, draft over target ids, draft_row, T) as the oracle walked them; needed
    to bound a differing final token (race_tie_bound).  Returns (n_decisions,
    near_tie_mismatches).  Raises AssertionError on a mismatch that is not explained by a
    near-tie (any mismatch when exact)."""
    B = acc.shape[0]
    if exact:
        assert np.array_equal(ref["accept_len"], acc)
        assert np.array_equal(ref["path"], path)
        assert np.array_equal(ref["emit"], emit)
        return int((ref["trace"][:, :, 3] > 0).sum()) + B, 0
    decisions = int((ref["trace"][:, :, 3] > 0).sum()) + B
    ties = 0
    for b in range(B):
        ra = int(ref["accept_len"][b])
        same = (ra == int(acc[b]) and np.array_equal(ref["path"][b], path[b])
                and np.array_equal(ref["emit"][b], emit[b]))
        if same:
            continue
        # first divergence along the path
        t = 0
        while t <= ra and t < path.shape[1] and ref["path"][b, t] == path[b, t]:
            t += 1
        if t > ra and ra == int(acc[b]):
            # same path, different final token: must be a near-tie of the race
            y, k1, y2, k2 = ref["race"][b]
            assert rows is not None, (f"sequence {b}: final token differs and no rows were "
                                      f"given to bound the race")
            v = int(ref["path"][b, ra])
            # v's rejected children: a tested node past v can only be v's child (at an
            # ancestor the children after the accepted one, itself at most v, are untried)
            n_rej = int(((ref["trace"][b, :, 3] == 2.0) &
                         (np.arange(ref["trace"].shape[1]) > v)).sum())
            bound = race_tie_bound(rows, b, v, n_rej, int(y), int(y2))
            assert k1 > 0 and (k1 - k2) / k1 < bound, (b, ref["race"][b], emit[b], bound)
            assert int(emit[b, ra]) == int(y2), (b, emit[b], ref["race"][b])
            ties += 1
            continue
        v = int(ref["path"][b, t - 1])
        tested = np.nonzero(ref["trace"][b, :, 3] > 0)[0]
        kids = [c for c in tested if c > v]
        near = [c for c in kids
                if abs(ref["trace"][b, c, 0] * ref["trace"][b, c, 1] - ref["trace"][b, c, 2])
                < NEAR_TIE_ABS]
        assert near, (f"sequence {b}: divergence at node {v} without a near-tie", ref["path"][b],
                      path[b], ref["emit"][b], emit[b])
        ties += 1
    return decisions, ties


def assert_tie_budget(decisions, ties):
    assert ties <= max(1, 1e-4 * decisions), (ties, decisions)


def attn_row_rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(got - ref).max(-1)
    den = np.maximum(np.abs(ref).max(-1), 1e-30)
    return num / den


# ---------------------------------------------------------------- EAGLE-2 expansion
CONF_RTOL = 1e-5      # draft confidences c (probabilities) against the oracle's fp64 ones
VALUE_RTOL = 1e-5     # path values V = prod c against the oracle's float32 products


def cand_id(level, s, j, k):
    """Candidate id of rank j under frontier slot s at `level` (EAGLE-2 numbering)."""
    return 1 + j if level == 1 else 1 + k + (level - 2) * k * k + s * k + j


def check_expansion(oracle, cand, out, ref_tok, ref_conf, k, D, n_out, own=None, tie_ok=None,
                    rows_for=None, slack=None):
    """Strict comparison of a GPU EAGLE-2 tree with the oracle, sequence by sequence.

    cand      the GPU tree state read back (eagle2_tree_candidates), numpy [B, C] arrays
    out       (tokens, parent, draft_row) the GPU wrote, numpy [B, n_out]
    ref_tok   oracle top-k tokens of every draft row, [B, R, k] (target ids)
    ref_conf  oracle softmax confidences of those tokens (fp64), [B, R, k]
    own       the oracle's own tree dict (eagle2_from_logits) or None
    tie_ok    tie_ok(b, r, tok_a, tok_b) -> True when the oracle's logits of the two tokens
              in row r are within the error of the logits the GPU ranked (only for rows the
              GPU computed itself); None: the GPU ranked the very same float32 logits, so
              its per-row top-k must equal the oracle's exactly.
    rows_for  the sequences whose rows ref_tok / ref_conf / own cover (default: all);
              the replay (check 2) runs for every sequence.
    slack     {b: s} for rows the GPU computed itself: s = 2 max |l_gpu - l_oracle| over the
              sequence's logits.  c = exp(l - m) / Z, so an error e_t in each logit moves
              c_t by at most |e_t| + max_s |e_s| relative; the confidence tolerance becomes
              CONF_RTOL + s and the value tolerance at level l VALUE_RTOL + l * s.

    Checks, for every sequence:
      1. per draft row the GPU expanded (its own frontier rows): the top-k tokens equal the
         oracle's (explained logit ties only, via tie_ok), confidences within CONF_RTOL;
      2. replay: the oracle's selection (Eagle2Tree) driven by the GPU's own tokens and
         confidences reproduces the GPU's parents, float32 path values (bit-exact),
         frontier slots / draft rows of every level and the reranked output, exactly;
      3. against the oracle's own tree (own): path values within VALUE_RTOL while the two
         trees share their frontiers; where they diverge, the first difference lies at a
         cut whose two candidates the oracle separates by less than the two sides' error
         (2 * VALUE_RTOL relative), or at a logit tie tie_ok explains.
    Returns dict(max_conf_rel, max_value_rel, tie_rows, tie_cuts, seqs_diff)."""
    import numpy as np
    tok_g, par_g, row_g = out
    B = tok_g.shape[0]
    stats = dict(max_conf_rel=0.0, max_value_rel=0.0, tie_rows=0, tie_cuts=0, seqs_diff=0,
                 max_slack=0.0 if slack is None else float(max(slack.values())))
    rows_for = set(range(B)) if rows_for is None else set(rows_for)
    for b in range(B):
        have = b in rows_for
        sl = 0.0 if slack is None else float(slack[b]) if have else 0.0
        rep = oracle.Eagle2Tree(k, D)
        for lvl in range(1, D + 1):
            k_in = 1 if lvl == 1 else k
            toks = np.zeros((k_in, k), np.int32)
            confs = np.zeros((k_in, k), np.float32)
            for s in range(k_in):
                par = rep.frontier[s]
                r = rep.row[par]
                ids = [cand_id(lvl, s, j, k) for j in range(k)]
                assert (cand["parent"][b, ids] == par).all(), (b, lvl, s)
                assert (cand["depth"][b, ids] == lvl).all(), (b, lvl, s)
                gt = cand["token"][b, ids]
                gc = cand["conf"][b, ids]
                toks[s], confs[s] = gt, gc
                if not have:
                    continue
                ot, oc = ref_tok[b][r], ref_conf[b][r]
                if not np.array_equal(gt, ot):
                    assert tie_ok is not None, (f"sequence {b} row {r}: top-k tokens differ on "
                                                f"identical logits", gt, ot)
                    j = int(np.nonzero(gt != ot)[0][0])
                    assert tie_ok(b, r, int(ot[j]), int(gt[j])), (b, r, gt, ot)
                    stats["tie_rows"] += 1
                for j in range(k):
                    hit = np.nonzero(ot == gt[j])[0]
                    if hit.size:
                        rel = abs(float(gc[j]) - oc[hit[0]]) / oc[hit[0]]
                        stats["max_conf_rel"] = max(stats["max_conf_rel"], rel)
                        assert rel <= CONF_RTOL + sl, (b, r, j, float(gc[j]), oc[hit[0]], sl)
            rep.expand(toks, confs)
            new = [cand_id(lvl, s, j, k) for s in range(k_in) for j in range(k)]
            gv = cand["value"][b, new]
            rv = np.array([rep.value[c] for c in new], np.float32)
            assert np.array_equal(gv.view(np.uint32), rv.view(np.uint32)), (b, lvl)
            if lvl < D:
                for s, c in enumerate(rep.frontier):
                    assert cand["draft_row"][b, c] == 1 + (lvl - 1) * k + s, (b, lvl, s)
        fin = rep.rerank(n_out)
        assert np.array_equal(fin["tokens"][1:], tok_g[b, 1:]), (b, fin["tokens"], tok_g[b])
        assert np.array_equal(fin["parent"], par_g[b]), (b, fin["parent"], par_g[b])
        assert np.array_equal(fin["draft_row"], row_g[b]), (b, fin["draft_row"], row_g[b])
        if own is None or not have:
            continue
        ot = own["trees"][b]
        if (np.array_equal(own["tokens"][b][1:], tok_g[b, 1:]) and
                np.array_equal(own["parent"][b], par_g[b]) and
                np.array_equal(own["draft_row"][b], row_g[b])):
            diverged = False
        else:
            diverged = True
            stats["seqs_diff"] += 1
        explained = False
        for lvl in range(1, D + 1):
            k_in = 1 if lvl == 1 else k
            new = [cand_id(lvl, s, j, k) for s in range(k_in) for j in range(k)]
            if any(ot.token[c] != rep.token[c] for c in new):
                # rows are the same (frontiers agreed so far): only a logit tie may differ
                assert tie_ok is not None, (b, lvl)
                explained = True
                break
            vtol = VALUE_RTOL + lvl * sl
            for c in new:
                rel = abs(float(rep.value[c]) - float(ot.value[c])) / float(ot.value[c])
                stats["max_value_rel"] = max(stats["max_value_rel"], rel)
                assert rel <= vtol, (b, lvl, c, rep.value[c], ot.value[c], vtol)
            fo, fg = ot.frontiers[lvl - 1], rep.frontiers[lvl - 1]
            if fo != fg:
                i = next(i for i in range(k) if fo[i] != fg[i])
                va, vg = float(ot.value[fo[i]]), float(ot.value[fg[i]])
                assert abs(va - vg) <= 2 * vtol * va, (
                    f"sequence {b}: level {lvl} frontier differs at slot {i} without a near-tie",
                    va, vg)
                stats["tie_cuts"] += 1
                explained = True
                break
        if not explained and diverged:
            # same candidates and values throughout: the global rerank cut decides
            key = lambda t, c: (-float(t.value[c]), t.depth[c], c)  # noqa: E731
            cands = [c for c in ot.value if c]
            lo = sorted(cands, key=lambda c: key(ot, c))[: n_out - 1]
            lg = sorted(cands, key=lambda c: key(rep, c))[: n_out - 1]
            vtol = VALUE_RTOL + D * sl
            for a, g in zip(lo, lg):
                if a != g:
                    va, vg = float(ot.value[a]), float(ot.value[g])
                    assert abs(va - vg) <= 2 * vtol * va, (
                        f"sequence {b}: rerank differs without a near-tie", va, vg)
            stats["tie_cuts"] += 1
    return stats
