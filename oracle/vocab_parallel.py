"""Vocab-parallel verify-and-accept walk on CPU ranks (oracle side).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: only the test suite may import it.

When the target and draft LM heads are split across ranks by vocabulary, each rank holds
a slice [v0, v1) of every logits row.  The walk of ``oracle.verify_accept`` (Lesson "推测
解码与 EAGLE-3", "不变量：Leviathan 拒绝采样" and steps 1-3; Guide "EAGLE-2" on tree
acceptance) then needs an exchange at exactly four points, the same ones at which the
GPU kernel's thread-block cluster exchanges through distributed shared memory:

  1. row statistics: each rank's (max z, sum exp(z - max)) over its slice, combined as
     M = max m_r, Z = sum Z_r exp(m_r - M), in rank order;
  2. the drafted token's probabilities q(x), p(x): only the rank owning x has them;
  3. a rejection's residual normaliser s = sum max(0, q_cur - p): a sum of the slices;
  4. the final token's exponential race argmax_t r_t / E_t: each rank's best (key,
     token), then the largest key, lower token on ties.

Everything between exchanges is the single-process walk restricted to the slice, in
double precision.  `comm` supplies all_gather of small float64 arrays (a thin wrapper
over torch.distributed in the tests).
"""
from __future__ import annotations

import math

import numpy as np

from . import race_sample, u_race, u_accept


def _stats(row, T):
    z = row.astype(np.float64) / T
    m = z.max() if z.size else -np.inf
    Z = float(np.exp(z - m).sum()) if np.isfinite(m) else 0.0
    return m, Z


def _combine_stats(pairs):
    """Rank-ordered combination of (m_r, Z_r)."""
    M = max(m for m, _ in pairs)
    return M, sum(Z * math.exp(m - M) for m, Z in pairs if np.isfinite(m))


def walk_sharded(comm, target, draft, tokens, parent, draft_row, v0, V, max_depth, T, seed, b):
    """One sequence's walk on this rank's vocabulary slice.

    target f32 [n, Vs], draft f32 [R, Vs]: the slice [v0, v0 + Vs) of every row of the
    sequence; tokens, parent, draft_row int [n] (whole-vocabulary token ids); b: the
    sequence's index (keys the uniforms).  T > 0.  Returns (accept_len, path, emit)
    like verify_accept."""
    n, Vs = target.shape
    has_child = np.zeros(n, bool)
    has_child[parent[1:]] = True
    mine = lambda t: v0 <= t < v0 + Vs          # noqa: E731
    v, a, path, emit = 0, 0, [0], []
    while True:
        mq, Zq = _combine_stats(comm.all_gather(np.array(_stats(target[v], T))))   # exchange 1
        q = np.exp(target[v].astype(np.float64) / T - mq) / Zq
        moved = False
        if has_child[v]:
            prow = draft[draft_row[v]]
            mp, Zp = _combine_stats(comm.all_gather(np.array(_stats(prow, T))))
            p = np.exp(prow.astype(np.float64) / T - mp) / Zp
            for c in range(v + 1, n):
                if parent[c] != v:
                    continue
                x = int(tokens[c])
                own = np.array([q[x - v0], p[x - v0]]) if mine(x) else np.zeros(2)
                qx, px = comm.all_gather(own).sum(axis=0)                         # exchange 2
                u = u_accept(seed, b, c)
                if px <= 0.0 or u < qx / px:
                    a += 1
                    path.append(c)
                    emit.append(x)
                    v = c
                    moved = True
                    break
                r = np.maximum(0.0, q - p)
                s = float(comm.all_gather(np.array([r.sum()]))[:, 0].sum())     # exchange 3
                if s > 0.0:
                    q = r / s
        if moved:
            continue
        # exchange 4: the race over this slice, then the best key across ranks
        full = np.zeros(V)
        full[v0:v0 + Vs] = q
        if (q > 0).any():
            y = race_sample(full, seed, b)
            key = q[y - v0] / -math.log(u_race(seed, b, 0, y))
            best = np.array([key, float(y)])
        else:
            best = np.array([-1.0, float(V)])
        allb = comm.all_gather(best)
        order = sorted(range(len(allb)), key=lambda r_: (-allb[r_][0], allb[r_][1]))
        y = int(allb[order[0]][1])
        emit.append(y)
        return a, path, emit
