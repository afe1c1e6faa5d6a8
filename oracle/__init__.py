"""CPU oracle for the EAGLE draft-tree verify-and-accept path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
CPU-baseline leg of the benchmark may import this package.  It shares no
code with the CUDA library: the numeric loops live in ``oracle.c`` (plain C,
double precision) and the tree bookkeeping of the EAGLE-2 expansion and
rerank lives here, in plain Python.

Pages cited (by title and section):
  [Lesson] "推测解码与 EAGLE-3" -- "不变量：Leviathan 拒绝采样", "什么决定加速",
           "KV cache 回滚", "动手构建" steps 1-6, "练习".
  [Guide]  "EAGLE-1/2/3 拆解" (txtmix.com) -- "无损性的来源与它的证明位置",
           "EAGLE-2：草稿树的 Expansion 与 Reranking", "一次 eagenerate 调用的完整流转".
  [TTT]    "EAGLE-3 完全拆解：Training-Time Test" -- "EAGLE-3 和 EAGLE-2 动态树如何拼在一起",
           "训练时的 attention mask 为什么要特殊处理".

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
something other than itself (published Philox known-answer vectors, the
closed form for the expected number of accepted tokens, chi-square tests of
losslessness, exact enumeration on tiny trees, library routines for
softmax / attention / matmul, brute force and invariants for the tree
selection).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

ORC_OK, ORC_BAD_TREE, ORC_BAD_TOKEN, ORC_NONFINITE, ORC_DEPTH, ORC_CAPACITY = 0, 1, 2, 4, 8, 16

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_D = ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_philox4x32_10.argtypes = [_P, _P, _P]
        L.orc_u_accept.argtypes = [_U64, _U32, _U32]
        L.orc_u_accept.restype = _D
        L.orc_u_race.argtypes = [_U64, _U32, _U32, _U32, _U32]
        L.orc_u_race.restype = _D
        L.orc_race_sample.argtypes = [_P, _I, _U64, _U32, _U32, _U32]
        L.orc_race_sample.restype = _I
        L.orc_tree_check.argtypes = [_P, _I, _P, _P]
        L.orc_tree_check.restype = _I
        L.orc_softmax_rows.argtypes = [_P, _I64, _I, _D, _P, _P, _P, _P]
        L.orc_verify_accept.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _D, _U64, _P,
                                        _P, _P, _P, _P, _P, _P]
        L.orc_sample_rows.argtypes = [_P, _I, _I, _I, _D, _U64, _P]
        L.orc_tree_attn.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _D, _P]
        L.orc_tree_attn.restype = _I
        L.orc_ttt_attn.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _D, _P]
        L.orc_ttt_attn.restype = _I
        L.orc_kv_compact.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I]
        L.orc_kv_compact.restype = _I
        L.orc_lmhead_rows.argtypes = [_P, _P, _I, _I, _I, _P, _I, _P]
        L.orc_row_topk.argtypes = [_P, _I64, _I, _I, _P, _P, _P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bf16_bits(t):
    """bf16 data as uint16 bit patterns (accepts a torch bf16 tensor or uint16 array)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- Philox
def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def u_accept(seed: int, b: int, node: int) -> float:
    return lib().orc_u_accept(seed, b, node)


def u_race(seed: int, b: int, c1: int, t: int, tag: int = 1) -> float:
    return lib().orc_u_race(seed, b, c1, t, tag)


def race_sample(r, seed: int, b: int, c1: int = 0, tag: int = 1) -> int:
    r = _c(r, np.float64)
    return lib().orc_race_sample(_ptr(r), r.size, seed, b, c1, tag)


# ---------------------------------------------------------------- tree
def tree_check(parent):
    """Ancestor bitmasks and depths of a parent array; None if invalid."""
    p = _c(parent, np.int32)
    anc = np.zeros(64, np.uint64)
    dep = np.zeros(64, np.int32)
    st = lib().orc_tree_check(_ptr(p), p.size, _ptr(anc), _ptr(dep))
    if st != ORC_OK:
        return None
    return anc[: p.size].copy(), dep[: p.size].copy()


# ---------------------------------------------------------------- softmax
def softmax_rows(logits, T: float):
    """(m, Z, argmax, status) per row of float32 logits, z = l / T."""
    x = _c(logits, np.float32)
    V = x.shape[-1]
    rows = x.size // V
    m = np.zeros(rows)
    Z = np.zeros(rows)
    am = np.zeros(rows, np.int32)
    st = np.zeros(rows, np.int32)
    lib().orc_softmax_rows(_ptr(x), rows, V, float(T), _ptr(m), _ptr(Z), _ptr(am), _ptr(st))
    shp = x.shape[:-1]
    return m.reshape(shp), Z.reshape(shp), am.reshape(shp), st.reshape(shp)


# ---------------------------------------------------------------- verify
def verify_accept(target, draft, tokens, parent, max_depth: int, T: float, seed: int,
                  draft_row=None, u_override=None):
    """Tree verify-and-accept walk (see oracle.c, walk_one).

    target f32 [B,n,V]; draft f32 [B,R,V]; tokens, parent i32 [B,n];
    draft_row i32 [B,n] or None (row i); u_override f64 [B,n] or None.
    """
    tgt = _c(target, np.float32)
    drf = _c(draft, np.float32)
    B, n, V = tgt.shape
    R = drf.shape[1]
    tok = _c(tokens, np.int32)
    par = _c(parent, np.int32)
    drow = None if draft_row is None else _c(draft_row, np.int32)
    uo = None if u_override is None else _c(u_override, np.float64)
    D = int(max_depth)
    out = dict(
        accept_len=np.zeros(B, np.int32),
        path=np.zeros((B, D + 1), np.int32),
        emit=np.zeros((B, D + 1), np.int32),
        trace=np.zeros((B, n, 4)),
        race=np.zeros((B, 4)),
        status=np.zeros(B, np.int32),
    )
    lib().orc_verify_accept(_ptr(tgt), _ptr(drf), _ptr(drow), _ptr(tok), _ptr(par), B, n, V, R, D,
                            float(T), int(seed) & (2**64 - 1), _ptr(uo),
                            _ptr(out["accept_len"]), _ptr(out["path"]), _ptr(out["emit"]),
                            _ptr(out["trace"]), _ptr(out["race"]), _ptr(out["status"]))
    return out


def d2t_scatter(draft, d2t, V: int):
    """Draft logits over a draft vocabulary of Vd tokens, f32 [..., Vd], placed in the
    target vocabulary of V tokens: draft id d sits at target id d + d2t[d], and every
    target id no draft id maps to gets -inf (probability 0).  This is what the draft
    distribution p is, as a function of target tokens, when the draft head has its own
    smaller vocabulary and the table d2t (int [Vd]) maps its outputs back (Guide,
    "EAGLE-3：取消特征约束…": the draft head ranks its own candidates and the table
    returns them to target ids).  The map must be one-to-one into [0, V)."""
    x = np.asarray(draft, np.float32)
    d2t = np.asarray(d2t, np.int64)
    Vd = x.shape[-1]
    assert d2t.shape == (Vd,)
    tgt_id = np.arange(Vd) + d2t
    assert tgt_id.min() >= 0 and tgt_id.max() < V, "d2t maps outside the target vocabulary"
    assert np.unique(tgt_id).size == Vd, "d2t maps two draft ids to one target id"
    full = np.full(x.shape[:-1] + (V,), -np.inf, np.float32)
    full[..., tgt_id] = x
    return full


def verify_accept_d2t(target, draft, d2t, tokens, parent, max_depth: int, T: float, seed: int,
                      draft_row=None, u_override=None):
    """verify_accept with draft rows over the draft vocabulary (f32 [B, R, Vd]) and the
    draft-to-target table d2t (int [Vd]); tokens are target ids.  p over the target
    vocabulary is the draft softmax at ids d + d2t[d] and 0 elsewhere (d2t_scatter);
    the walk is then the one of verify_accept, unchanged."""
    V = np.asarray(target).shape[-1]
    return verify_accept(target, d2t_scatter(draft, d2t, V), tokens, parent, max_depth, T, seed,
                         draft_row=draft_row, u_override=u_override)


def filter_logits(logits, T: float, top_k: int = 0, top_p: float = 0.0):
    """Top-k then top-p filtering of rows of logits at temperature T > 0, as logits:
    kept entries unchanged, the others -inf (probability 0 after the softmax).

    Guide, "一次 eagenerate 调用的完整流转": eagenerate takes temperature, top_p and
    top_k (0 = off).  Reading, where the pages are silent: rank a row's tokens by
    probability (logit desc, lower token first on ties); top-k keeps the first k;
    top-p then keeps the shortest prefix of that order whose probability, renormalised
    over what top-k kept, reaches top_p (at least one token; top_p <= 0 or >= 1 keeps
    all).  Applied the same way to the target rows (q) and the draft rows (p)."""
    x = np.asarray(logits, np.float32)
    V = x.shape[-1]
    flat = x.reshape(-1, V)
    out = np.full_like(flat, -np.inf)
    for r in range(flat.shape[0]):
        row = flat[r].astype(np.float64)
        order = np.lexsort((np.arange(V), -row))          # logit desc, then token asc
        keep = V if top_k <= 0 else min(int(top_k), V)
        if 0.0 < top_p < 1.0:
            z = row[order[:keep]] / T
            pr = np.exp(z - z.max())
            cum = np.cumsum(pr) / pr.sum()
            keep = min(keep, int(np.searchsorted(cum, top_p, side="left")) + 1)
        idx = np.array(order[:keep])
        out[r, idx] = flat[r, idx]
    return out.reshape(x.shape)


def verify_accept_filtered(target, draft, tokens, parent, max_depth: int, T: float, seed: int,
                           top_k: int = 0, top_p: float = 0.0, draft_row=None, u_override=None):
    """verify_accept with q and p replaced by their top-k / top-p filtered versions
    (filter_logits, the same filter for both); the walk itself is unchanged."""
    if T > 0:
        target = filter_logits(target, T, top_k, top_p)
        draft = filter_logits(draft, T, top_k, top_p)
    return verify_accept(target, draft, tokens, parent, max_depth, T, seed, draft_row=draft_row,
                         u_override=u_override)


def sample_rows(logits, T: float, seed: int):
    """One token per row of logits [B, rows, V] from softmax(row / T) (argmax at T = 0)."""
    x = _c(logits, np.float32)
    B, rows, V = x.shape
    out = np.zeros((B, rows), np.int32)
    lib().orc_sample_rows(_ptr(x), B, rows, V, float(T), int(seed) & (2**64 - 1), _ptr(out))
    return out


# ---------------------------------------------------------------- attention
def tree_attn(q, k, v, kv_len, parent, scale: float):
    """Tree-masked GQA attention in double.  q [B,n,Hq,d], k/v [B,Hkv,Lmax,d] (bf16)."""
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    B, n, Hq, d = qb.shape
    Hkv, Lmax = kb.shape[1], kb.shape[2]
    kl = _c(kv_len, np.int32)
    par = _c(parent, np.int32)
    out = np.zeros((B, n, Hq, d))
    st = lib().orc_tree_attn(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(kl), _ptr(par), B, n, Hq, Hkv, d,
                             Lmax, float(scale), _ptr(out))
    if st != ORC_OK:
        raise ValueError(f"tree_attn: invalid input (status {st})")
    return out


def ttt_attn(q, k, v, r: int, scale: float):
    """Training-time-test attention of the queries of round r in double (see oracle.c,
    orc_ttt_attn).  q [B,S,Hq,d], k/v [B,Hkv,R1,S,d] (bf16; round 0 = original tokens)."""
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    B, S, Hq, d = qb.shape
    Hkv, R1 = kb.shape[1], kb.shape[2]
    if kb.shape != (B, Hkv, R1, S, d) or vb.shape != kb.shape:
        raise ValueError("ttt_attn: k / v must be [B, Hkv, R1, S, d]")
    out = np.zeros((B, S, Hq, d))
    st = lib().orc_ttt_attn(_ptr(qb), _ptr(kb), _ptr(vb), B, S, Hq, Hkv, d, R1, int(r),
                            float(scale), _ptr(out))
    if st != ORC_OK:
        raise ValueError(f"ttt_attn: invalid input (status {st})")
    return out


# ---------------------------------------------------------------- compaction
def kv_compact(k_bits, v_bits, kv_len, path, accept_len, max_depth: int):
    """In-place compaction of uint16 K/V caches [n_layers,B,Hkv,Lmax,d]; updates kv_len."""
    assert k_bits.dtype == np.uint16 and k_bits.flags.c_contiguous
    assert v_bits.dtype == np.uint16 and v_bits.flags.c_contiguous
    assert kv_len.dtype == np.int32 and kv_len.flags.c_contiguous
    nl, B, Hkv, Lmax, d = k_bits.shape
    p = _c(path, np.int32)
    a = _c(accept_len, np.int32)
    return lib().orc_kv_compact(_ptr(k_bits), _ptr(v_bits), _ptr(kv_len), _ptr(p), _ptr(a),
                                nl, B, Hkv, d, Lmax, int(max_depth))


# ---------------------------------------------------------------- LM head, top-k
def lmhead_rows(hidden, w, rows):
    """logits[rows] = hidden[rows] . W^T in double.  hidden [M,K], w [N,K] (bf16)."""
    hb, wb = _bf16_bits(hidden), _bf16_bits(w)
    M, K = hb.shape
    N = wb.shape[0]
    r = _c(rows, np.int32)
    out = np.zeros((r.size, N))
    lib().orc_lmhead_rows(_ptr(hb), _ptr(wb), M, K, N, _ptr(r), r.size, _ptr(out))
    return out


def row_topk(logits, k: int):
    """Top-k tokens (logit desc, token asc) and their softmax confidences (double)."""
    x = _c(logits, np.float32)
    V = x.shape[-1]
    rows = x.size // V
    tok = np.zeros((rows, k), np.int32)
    conf = np.zeros((rows, k))
    st = np.zeros(rows, np.int32)
    lib().orc_row_topk(_ptr(x), rows, V, k, _ptr(tok), _ptr(conf), _ptr(st))
    shp = x.shape[:-1] + (k,)
    return tok.reshape(shp), conf.reshape(shp), st.reshape(x.shape[:-1])


# ---------------------------------------------------------------- EAGLE-2 tree
def draft_rows(top_k: int, depth: int) -> int:
    """Draft-logit rows per sequence: the root plus top_k frontier rows for levels 2..depth."""
    return 1 + (depth - 1) * top_k


def level_row_offset(level: int, top_k: int) -> int:
    """First draft row read at expansion level `level` (1-based)."""
    return 0 if level == 1 else 1 + (level - 2) * top_k


class Eagle2Tree:
    """EAGLE-2 expansion and reranking for one sequence.

    Guide, "EAGLE-2：草稿树的 Expansion 与 Reranking": the value of node t_i is the
    product of draft confidences along the root-to-t_i path (V_i = prod c_j, the
    draft being well calibrated, section "一个可核对的经验性质"); the expansion stage
    runs, level by level, the draft forward only on the k nodes of the previous
    level with the highest V; the reranking stage orders every node of the tree
    by V and sends the global top-N to verification (a shallow unexpanded node may
    beat a deep expanded one).  Depth and k are fixed.  TTT page, "EAGLE-3 和
    EAGLE-2 动态树如何拼在一起", restates V_i and the per-level choice of 10 nodes.

    Readings where the pages are silent:
      * confidences are the temperature-1 softmax of the draft logits;
      * level 1 expands the root's row into its top-k tokens; each later level
        expands the k frontier nodes, each into its top-k tokens, giving k*k
        candidates of which the k with the largest V (lower candidate id on ties)
        form the next frontier;
      * V products are taken in float32 (the precision of the kernel, since the
        comparison of V values decides which nodes are kept); the root has V = 1;
      * rerank keeps the root plus the n-1 candidates that come first by
        (V desc, depth asc, id asc); since c <= 1 a parent is never ranked after
        its child, so the kept set is ancestor-closed; output order is
        topological: (depth asc, V desc, id asc).
    Candidate ids: root 0; level 1: 1 + j (j = rank in the root's top-k);
    level l >= 2: 1 + k + (l-2) k^2 + s k + j (s = frontier slot, j = rank).
    Draft rows: root -> 0; the frontier slot s chosen at level l (l < depth)
    is expanded at level l+1 from row 1 + (l-1) k + s.
    """

    def __init__(self, top_k: int, depth: int):
        self.k = top_k
        self.D = depth
        self.value = {0: np.float32(1.0)}
        self.parent = {0: -1}
        self.token = {0: -1}
        self.depth = {0: 0}
        self.row = {0: 0}
        self.frontier = [0]
        self.level = 0
        self.frontiers = []

    def expand(self, tok, conf32):
        """One level.  tok i32 [k_in, k], conf32 f32 [k_in, k] for the current frontier rows."""
        k = self.k
        self.level += 1
        lvl = self.level
        tok = np.asarray(tok, np.int32)
        conf32 = np.asarray(conf32, np.float32)
        assert tok.shape == (len(self.frontier), k)
        new = []
        for s, par in enumerate(self.frontier):
            for j in range(k):
                cid = 1 + j if lvl == 1 else 1 + k + (lvl - 2) * k * k + s * k + j
                self.value[cid] = np.float32(self.value[par] * conf32[s, j])
                self.parent[cid] = par
                self.token[cid] = int(tok[s, j])
                self.depth[cid] = lvl
                new.append(cid)
        order = sorted(new, key=lambda c: (-float(self.value[c]), c))
        self.frontier = order[:k]
        self.frontiers.append(list(self.frontier))
        if lvl < self.D:
            for s, c in enumerate(self.frontier):
                self.row[c] = 1 + (lvl - 1) * k + s
        return self.frontier

    def rerank(self, n_out: int, root_token: int = -1):
        cands = [c for c in self.value if c != 0]
        top = sorted(cands, key=lambda c: (-float(self.value[c]), self.depth[c], c))[: n_out - 1]
        nodes = [0] + sorted(top, key=lambda c: (self.depth[c], -float(self.value[c]), c))
        index = {c: i for i, c in enumerate(nodes)}
        tokens = np.array([root_token] + [self.token[c] for c in nodes[1:]], np.int32)
        parent = np.array([-1] + [index[self.parent[c]] for c in nodes[1:]], np.int32)
        row = np.array([self.row.get(c, -1) for c in nodes], np.int32)
        values = np.array([self.value[c] for c in nodes], np.float32)
        return dict(tokens=tokens, parent=parent, draft_row=row, cand=np.array(nodes, np.int32),
                    value=values)


def eagle2_from_logits(logits, top_k: int, depth: int, n_out: int, root_tokens=None, d2t=None):
    """Whole expansion + rerank from per-row draft logits f32 [B, R, V] (R = draft_rows).
    With d2t (int [V]), the rows are over a draft vocabulary and each chosen draft id d
    enters the tree as the target id d + d2t[d]; the ranking (top-k by logit, ties to the
    lower draft id) and the values are those of the draft vocabulary."""
    x = _c(logits, np.float32)
    B, R, V = x.shape
    assert R >= draft_rows(top_k, depth)
    if d2t is not None:
        d2t = np.asarray(d2t, np.int64)
        assert d2t.shape == (V,)
    trees = [Eagle2Tree(top_k, depth) for _ in range(B)]
    for lvl in range(1, depth + 1):
        off = level_row_offset(lvl, top_k)
        k_in = 1 if lvl == 1 else top_k
        tok, conf, st = row_topk(x[:, off:off + k_in], top_k)
        if d2t is not None:
            tok = (tok + d2t[tok]).astype(np.int32)
        for b in range(B):
            trees[b].expand(tok[b], conf[b].astype(np.float32))
    outs = [t.rerank(n_out, -1 if root_tokens is None else int(root_tokens[b]))
            for b, t in enumerate(trees)]
    res = {key: np.stack([o[key] for o in outs]) for key in outs[0]}
    res["trees"] = trees
    return res


# ---------------------------------------------------------------- static trees
def static_tree_from_choices(choices):
    """A static draft tree (EAGLE-1 / Medusa style) from its list of choices: each choice
    is a path of child ranks from the root, (r_1, ..., r_d), naming the node reached by
    taking, at each depth, the r-th best token of the parent's draft distribution.
    Guide, "EAGLE-2：草稿树的 Expansion 与 Reranking" (the static trees EAGLE-2 replaces
    add a fixed k candidates per step) and the file layout it points to (choices.py).

    Readings where the pages are silent: every proper prefix of a choice must itself
    be a choice (a node's parent is in the tree); choices are distinct and ranks are
    >= 0.  Node order: the root (node 0), then the choices sorted by (length,
    lexicographic) -- a topological order.  The children of a node are drafted from
    one draft row: internal nodes (nodes with children) are numbered 0, 1, ... in node
    order, and that number is the node's draft row.
    Returns dict(parent, rank, depth, draft_row) int32 [n] (root: parent -1, rank -1)."""
    paths = [tuple(int(r) for r in c) for c in choices]
    if len(set(paths)) != len(paths):
        raise ValueError("duplicate choice")
    if any(len(c) == 0 or min(c) < 0 for c in paths):
        raise ValueError("empty choice or negative rank")
    have = set(paths)
    for c in paths:
        if len(c) > 1 and c[:-1] not in have:
            raise ValueError(f"choice {c} without its parent {c[:-1]}")
    order = sorted(paths, key=lambda c: (len(c), c))
    index = {(): 0}
    for i, c in enumerate(order):
        index[c] = i + 1
    n = len(order) + 1
    parent = np.full(n, -1, np.int32)
    rank = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int32)
    for c in order:
        i = index[c]
        parent[i] = index[c[:-1]]
        rank[i] = c[-1]
        depth[i] = len(c)
    has_kids = np.zeros(n, bool)
    has_kids[parent[1:]] = True
    draft_row = np.full(n, -1, np.int32)
    draft_row[has_kids] = np.arange(int(has_kids.sum()), dtype=np.int32)
    return dict(parent=parent, rank=rank, depth=depth, draft_row=draft_row)


def static_tree_tokens(logits, tree):
    """Tokens of a static tree's nodes from the draft rows of its internal nodes,
    f32 [B, R, V] (row draft_row[v] holds the distribution after node v): node i takes
    the rank[i]-th best token (logit desc, token asc) of its parent's row.  The root's
    token is -1 (it is the last committed token, known to the caller)."""
    x = _c(logits, np.float32)
    B, R, V = x.shape
    par, rank, drow = tree["parent"], tree["rank"], tree["draft_row"]
    K = int(rank.max()) + 1 if len(rank) > 1 else 1
    tok, _, st = row_topk(x, K)
    out = np.full((B, len(par)), -1, np.int32)
    for i in range(1, len(par)):
        out[:, i] = tok[:, drow[par[i]], rank[i]]
    return out
