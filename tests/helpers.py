"""Comparison helpers shared by the GPU parity tests.

Tolerances (written out here and in each test):
  * integer / index results: bit-exact;
  * temperature 0: bit-exact (decisions compare raw float32 logits on both sides);
  * temperature > 0: accept decisions identical except near-ties, a tested child
    with |u * p(x) - q_cur(x)| < 1e-6 (probabilities from the double-precision
    oracle), or a sampling race whose two best keys differ by less than 1e-5
    relative; the near-tie count must stay below 1e-4 of all decisions (one is
    tolerated in small runs);
  * probabilities / softmax statistics: 1e-5 relative;
  * bf16 attention output: per (sequence, node, head) row,
    max |O_gpu - O_ref| / max |O_ref| <= 1e-2.
"""
from __future__ import annotations

import numpy as np

NEAR_TIE_ABS = 1e-6
RACE_TIE_REL = 1e-5


def compare_walks(ref, acc, path, emit, exact=False):
    """Compare the GPU walk (acc, path, emit numpy arrays) with the oracle's.

    Returns (n_decisions, near_tie_mismatches).  Raises AssertionError on a
    mismatch that is not explained by a near-tie (any mismatch when exact)."""
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
            assert k1 > 0 and (k1 - k2) / k1 < RACE_TIE_REL, (b, ref["race"][b], emit[b])
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
