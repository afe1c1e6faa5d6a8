"""The library's static-tree planner (host code in the .so, no GPU) against the oracle.

Static trees (EAGLE-1 / Medusa style): Guide "EAGLE-2：草稿树的 Expansion 与 Reranking".
"""
import numpy as np
import pytest

import oracle
import workloads as W


def _E():
    import eagle_tree_speculative_gb300 as E
    return E


def _random_choices(seed, cap=50):
    g = W.rng(seed, 49)
    choices, frontier = set(), [()]
    while frontier and len(choices) < cap:
        c = frontier.pop(0)
        for r in range(int(g.integers(0, 5))):
            if len(choices) < cap:
                choices.add(c + (r,))
                frontier.append(c + (r,))
    return sorted(choices, key=lambda c: g.random())


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_planner_matches_oracle(seed):
    choices = _random_choices(seed)
    got = _E().eagle_static_tree(choices)
    ref = oracle.static_tree_from_choices(choices)
    for key in ("parent", "rank", "depth", "draft_row"):
        assert np.array_equal(got[key], ref[key]), key


def test_planner_rejects_bad_choice_lists():
    E = _E()
    for bad in ([(0,), (0,)], [(1, 0)], [(0,), (16,)], [(0,)] + [(0, 1, 2, 3)]):
        with pytest.raises(RuntimeError):
            E.eagle_static_tree(bad)
    with pytest.raises(RuntimeError):                # 64 nodes at most
        E.eagle_static_tree([(i % 16,) if i < 16 else (i // 16 - 1, i % 16) for i in range(70)])
