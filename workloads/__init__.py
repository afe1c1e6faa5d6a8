"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module holds no arithmetic of the method: it draws normal variates,
random tree shapes and bf16 roundings, and assembles arrays by index.  The
random numbers the method itself draws (accept uniforms, sampling races) are
NOT generated here; the CUDA library and the oracle each implement Philox.

Every array is keyed per sequence (numpy's Philox bit generator seeded with
SeedSequence([seed, tag, b, ...])), so any single sequence of a large batch
can be regenerated on its own.

Workload shapes follow the pages' setups: Vicuna-13B (40 heads, V = 32000),
Llama-3-8B (32 q / 8 kv heads, V = 128256, hidden 4096) and Llama-70B
(64 q / 8 kv heads); trees of 60 / 48 nodes, depth 6 (EAGLE-2) or 8 (EAGLE-3),
10 nodes expanded per level (Guide "EAGLE-2：草稿树的 Expansion 与 Reranking",
TTT page "EAGLE-3 和 EAGLE-2 动态树如何拼在一起").  The pages measure on public
chat/code/math benchmarks; none is used or reproduced here: these synthetic
logits, hidden states and caches stand in for them.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Stream tags.
TAG_TARGET = 3        # target logits rows
TAG_DRAFT_NOISE = 4   # draft = target + sigma * noise
TAG_LEAF = 5          # target rows of tree leaves that were never expanded
TAG_Q, TAG_K, TAG_V = 6, 7, 8
TAG_HIDDEN = 9
TAG_W = 10
TAG_TREE = 11
TAG_CACHE = 12
TAG_CHAIN = 13
TAG_D2T = 14          # which target ids a draft vocabulary holds
TAG_TTT_Q, TAG_TTT_K, TAG_TTT_V = 15, 16, 17   # training-time-test attention


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    n: int                 # tree nodes including the root
    depth: int
    top_k: int
    V: int
    sigma: float           # draft-logit noise
    target_std: float = 2.0
    T: tuple = (1.0,)
    Hq: int = 0
    Hkv: int = 0
    head_dim: int = 128
    L: int = 0             # committed KV length
    H: int = 0             # hidden size (draft LM head)
    w_std: float = 0.02
    n_layers: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return 1 + (self.depth - 1) * self.top_k

    @property
    def Lmax(self) -> int:
        return self.L + self.n


CONFIGS = {
    # chain verify, B=1: root + 5 drafts, V=32000, T=1 and T=0, 1000 independent steps
    "chain": Config("chain", B=1, n=6, depth=5, top_k=1, V=32000, sigma=0.5, T=(1.0, 0.0),
                    extra={"steps": 1000}),
    # EAGLE-2 tree, B=1, Vicuna-13B shape
    "eagle2_b1": Config("eagle2_b1", B=1, n=60, depth=6, top_k=10, V=32000, sigma=0.5,
                        T=(0.0, 1.0), Hq=40, Hkv=40, L=2048),
    # EAGLE-3 tree, B=64, Llama-3-8B shape, 32-layer compaction
    "eagle3_b64": Config("eagle3_b64", B=64, n=60, depth=8, top_k=10, V=128256, sigma=0.3,
                         T=(1.0,), Hq=32, Hkv=8, L=4096, H=4096, n_layers=32),
    # draft expansion, Llama-3-8B shape: 64 seqs x 10 frontier rows, 8 levels, rerank to 60
    "expand_b64": Config("expand_b64", B=64, n=60, depth=8, top_k=10, V=128256, sigma=0.3,
                         H=4096),
    # sweep, Llama-70B shape
    "sweep_70b": Config("sweep_70b", B=64, n=48, depth=6, top_k=10, V=128256, sigma=0.5,
                        T=(0.0, 1.0), Hq=64, Hkv=8, L=4096,
                        extra={"B": (1, 8, 32, 64), "L": (512, 1024, 2048, 4096, 8192, 16384, 32768),
                               "V": (32000, 128256), "sigma": (0.1, 0.5, 1.0)}),
}


def rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), *map(int, key)])))


def normal(shape, std: float, seed: int, *key: int) -> np.ndarray:
    return rng(seed, *key).standard_normal(shape, dtype=np.float32) * np.float32(std)


def per_seq_normal(B: int, row_shape, std: float, seed: int, tag: int, threads: int = 8) -> np.ndarray:
    """[B, *row_shape] float32, sequence b drawn from its own stream (seed, tag, b)."""
    out = np.empty((B, *row_shape), np.float32)

    def fill(b):
        g = rng(seed, tag, b)
        g.standard_normal(row_shape, dtype=np.float32, out=out[b])
        if std != 1.0:
            out[b] *= np.float32(std)

    with ThreadPoolExecutor(max_workers=max(1, min(threads, B))) as ex:
        list(ex.map(fill, range(B)))
    return out


def to_bf16(x: np.ndarray):
    """Round float32 to bfloat16 (round-to-nearest-even) as a torch CPU tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)


# ---------------------------------------------------------------- trees
def chain_tree(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def random_tree(n: int, max_depth: int, seed: int, *key: int) -> np.ndarray:
    """A random parent array (parent[0] = -1, parent[i] < i) of depth <= max_depth."""
    g = rng(seed, TAG_TREE, *key)
    parent = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int32)
    for i in range(1, n):
        ok = np.nonzero(depth[:i] < max_depth)[0]
        pa = int(ok[g.integers(len(ok))])
        parent[i] = pa
        depth[i] = depth[pa] + 1
    return parent


def random_tokens(B: int, n: int, V: int, seed: int) -> np.ndarray:
    t = rng(seed, TAG_TREE, 1 << 20).integers(0, V, size=(B, n), dtype=np.int32)
    t[:, 0] = -1
    return t


# ---------------------------------------------------------------- verify inputs
def chain_logits(B: int, n: int, V: int, sigma: float, target_std: float, seed: int):
    """Chain config: target rows ~ N(0, target_std^2), draft = target + N(0, sigma^2).

    Row i of both is the distribution after node i (node 0 = root)."""
    tgt = per_seq_normal(B, (n, V), target_std, seed, TAG_TARGET)
    drf = tgt + per_seq_normal(B, (n, V), sigma, seed, TAG_DRAFT_NOISE)
    return tgt, drf


def tree_draft_rows(cfg: Config, seed: int, B: int | None = None, V: int | None = None,
                    sigma: float | None = None):
    """Per draft row r: the target row T_r and the draft row T_r + sigma * noise."""
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    sigma = cfg.sigma if sigma is None else sigma
    trow = per_seq_normal(B, (cfg.R, V), cfg.target_std, seed, TAG_TARGET)
    drows = trow + per_seq_normal(B, (cfg.R, V), sigma, seed, TAG_DRAFT_NOISE)
    return trow, drows


def d2t_table(V: int, Vd: int, seed: int):
    """A draft vocabulary of Vd target ids, a sorted seeded subset of [0, V), as the
    table d2t (int32 [Vd], draft id d -> target id d + d2t[d]) and the ids themselves."""
    ids = np.sort(rng(seed, TAG_D2T, V, Vd).choice(V, size=Vd, replace=False))
    return (ids - np.arange(Vd)).astype(np.int32), ids.astype(np.int64)


def tree_draft_rows_d2t(cfg: Config, seed: int, ids: np.ndarray, B: int | None = None,
                        V: int | None = None, sigma: float | None = None):
    """Per draft row r: the target row T_r over V ids, and the draft row over the draft
    vocabulary (the entries of T_r at the vocabulary's ids, plus sigma * noise)."""
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    sigma = cfg.sigma if sigma is None else sigma
    trow = per_seq_normal(B, (cfg.R, V), cfg.target_std, seed, TAG_TARGET)
    drows = trow[..., ids] + per_seq_normal(B, (cfg.R, len(ids)), sigma, seed, TAG_DRAFT_NOISE)
    return trow, drows.astype(np.float32)


def assemble_target(trow: np.ndarray, draft_row: np.ndarray, cand: np.ndarray,
                    target_std: float, seed: int) -> np.ndarray:
    """Target logits per tree node: the row's own target row if the node was expanded,
    else a fresh row keyed by (sequence, candidate id)."""
    B, R, V = trow.shape
    n = draft_row.shape[1]
    out = np.empty((B, n, V), np.float32)
    for b in range(B):
        for i in range(n):
            r = int(draft_row[b, i])
            if r >= 0:
                out[b, i] = trow[b, r]
            else:
                out[b, i] = normal(V, target_std, seed, TAG_LEAF, b, int(cand[b, i]))
    return out


# ---------------------------------------------------------------- attention / cache
def attn_inputs(B: int, n: int, Hq: int, Hkv: int, d: int, kv_len, Lmax: int, seed: int):
    """q [B,n,Hq,d], k/v [B,Hkv,Lmax,d] (bf16, ~N(0,1)), kv_len int32 [B]."""
    kv_len = np.broadcast_to(np.asarray(kv_len, np.int32), (B,)).copy()
    q = to_bf16(per_seq_normal(B, (n, Hq, d), 1.0, seed, TAG_Q))
    k = to_bf16(per_seq_normal(B, (Hkv, Lmax, d), 1.0, seed, TAG_K))
    v = to_bf16(per_seq_normal(B, (Hkv, Lmax, d), 1.0, seed, TAG_V))
    return q, k, v, kv_len


def ttt_inputs(B: int, S: int, Hq: int, Hkv: int, d: int, R1: int, seed: int):
    """Training-time-test attention inputs: q [B,S,Hq,d] (the queries of one round) and
    k / v [B,Hkv,R1,S,d] (round 0 = the original tokens, then the simulated rounds), bf16
    ~N(0,1)."""
    q = to_bf16(per_seq_normal(B, (S, Hq, d), 1.0, seed, TAG_TTT_Q))
    k = to_bf16(per_seq_normal(B, (Hkv, R1, S, d), 1.0, seed, TAG_TTT_K))
    v = to_bf16(per_seq_normal(B, (Hkv, R1, S, d), 1.0, seed, TAG_TTT_V))
    return q, k, v


def kv_cache(n_layers: int, B: int, Hkv: int, Lmax: int, d: int, seed: int):
    """K and V caches [n_layers,B,Hkv,Lmax,d] as bf16 tensors with distinct random rows."""
    k = to_bf16(np.stack([normal((B, Hkv, Lmax, d), 1.0, seed, TAG_CACHE, l, 0)
                          for l in range(n_layers)]))
    v = to_bf16(np.stack([normal((B, Hkv, Lmax, d), 1.0, seed, TAG_CACHE, l, 1)
                          for l in range(n_layers)]))
    return k, v


# ---------------------------------------------------------------- draft LM head
def lm_head(V: int, H: int, std: float, seed: int, block: int = 4096, threads: int = 8):
    """W [V, H] bf16 ~ N(0, std^2), generated in row blocks keyed (seed, TAG_W, block)."""
    import torch
    out = torch.empty((V, H), dtype=torch.bfloat16)
    nb = (V + block - 1) // block

    def fill(i):
        r0, r1 = i * block, min(V, (i + 1) * block)
        out[r0:r1] = to_bf16(normal((r1 - r0, H), std, seed, TAG_W, i))

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(nb)))
    return out


def hidden_states(B: int, k_in: int, H: int, level: int, seed: int):
    """Draft hidden states for one expansion level: [B, k_in, H] bf16 ~ N(0,1), keyed (b, level)."""
    return to_bf16(np.stack([normal((k_in, H), 1.0, seed, TAG_HIDDEN, b, level) for b in range(B)]))
