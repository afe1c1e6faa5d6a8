"""GB300 (sm_103a) draft-tree verify-and-accept for EAGLE-style speculative decoding.

Thin binding over the C ABI of include/eagle.h: every function marshals torch
CUDA tensors into device pointers plus the current CUDA stream and calls the
library entry point of the same name; all arithmetic runs in the library's
kernels.  PyTorch only provides device memory and streams.  Functions raise
EagleError on a non-OK status; errors found in device data are reported through
the optional ``dev_status`` int32 tensor (bits EAGLE_DEV_*).
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib

EAGLE_DEV_BAD_TREE = 0x01
EAGLE_DEV_BAD_TOKEN = 0x02
EAGLE_DEV_NONFINITE = 0x04
EAGLE_DEV_DEPTH = 0x08
EAGLE_DEV_CAPACITY = 0x10
EAGLE_DEV_TIMEOUT = 0x20


class EagleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {_lib.load().eagle_status_str(code).decode()} ({code})")


def lib():
    return _lib.load()


def _check(fn: str, code: int):
    if code != 0:
        raise EagleError(fn, code)


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _dev_or_pinned(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    """A CUDA tensor, or a page-locked host tensor, which the GPU reads in place over
    unified addressing (the kernel then moves only the bytes it touches)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t
    return _dev(t, name, dtype)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _status(dev_status, device):
    if dev_status is None:
        return None
    return _dev(dev_status, "dev_status", torch.int32)


# ---------------------------------------------------------------- workspace sizes
def tree_attn_workspace_size(B, n, Hq, Hkv, head_dim, Lmax) -> int:
    return int(lib().eagle_tree_attn_workspace_size(B, n, Hq, Hkv, head_dim, Lmax))


def tree_state_size(B, top_k, depth) -> int:
    return int(lib().eagle2_tree_state_size(B, top_k, depth))


# ---------------------------------------------------------------- calls
def eagle_tree_attn(q, k_cache, v_cache, kv_len, parent, scale=None, out=None, workspace=None,
                    dev_status=None, stream=None):
    """q [B,n,Hq,d], k/v cache [B,Hkv,Lmax,d] bf16; kv_len [B], parent [B,n] int32."""
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.bfloat16)
    _dev(v_cache, "v_cache", torch.bfloat16)
    _dev(kv_len, "kv_len", torch.int32)
    _dev(parent, "parent", torch.int32)
    B, n, Hq, d = q.shape
    Hkv, Lmax = k_cache.shape[-3], k_cache.shape[-2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.bfloat16)
    need = tree_attn_workspace_size(B, n, Hq, Hkv, d, Lmax)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("eagle_tree_attn", lib().eagle_tree_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(parent), _ptr(out),
        B, n, Hq, Hkv, d, Lmax, float(scale), _ptr(workspace), ws_bytes,
        _ptr(_status(dev_status, q.device)), _stream(stream)))
    return out


def eagle_ttt_attn(q, k, v, r, scale=None, out=None, dev_status=None, stream=None):
    """Training-time-test attention of the queries of round r.  q [B,S,Hq,d] and
    k / v [B,Hkv,R1,S,d] bf16 (round 0 = the original tokens); returns out [B,S,Hq,d]."""
    _dev(q, "q", torch.bfloat16)
    _dev(k, "k", torch.bfloat16)
    _dev(v, "v", torch.bfloat16)
    B, S, Hq, d = q.shape
    if k.dim() != 5 or tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != S \
            or k.shape[4] != d:
        raise ValueError("eagle_ttt_attn: k / v must be [B, Hkv, R1, S, d] matching q")
    Hkv, R1 = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.bfloat16)
    _check("eagle_ttt_attn", lib().eagle_ttt_attn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, Hq, Hkv, d, R1, int(r), float(scale),
        _ptr(_status(dev_status, q.device)), _stream(stream)))
    return out


def verify_filter_workspace_size(B, n, R) -> int:
    return int(lib().eagle_verify_filter_workspace_size(B, n, R))


def eagle_d2t_inverse(d2t, V, t2d=None, dev_status=None, stream=None):
    """t2d int32 [V]: the draft id of each target id (d + d2t[d] -> d), -1 where none."""
    _dev(d2t, "d2t", torch.int32)
    t2d = torch.empty(V, dtype=torch.int32, device=d2t.device) if t2d is None else t2d
    _dev(t2d, "t2d", torch.int32)
    _check("eagle_d2t_inverse", lib().eagle_d2t_inverse(
        _ptr(d2t), d2t.numel(), int(V), _ptr(t2d), _ptr(_status(dev_status, d2t.device)),
        _stream(stream)))
    return t2d


def eagle_verify_accept(target_logits, draft_logits, tokens, parent, max_depth, temperature, seed,
                        draft_row=None, accept_len=None, path=None, emit=None, row_stats=None,
                        dev_status=None, stream=None, t2d=None, top_k=0, top_p=0.0,
                        workspace=None):
    """Returns (accept_len [B], path [B,D+1], emit [B,D+1]) int32 tensors.  With t2d
    (from eagle_d2t_inverse) the draft rows are over the draft vocabulary
    [B, R, Vd] and tokens are target ids.  target_logits may be a pinned host tensor:
    the walk then reads only the rows it visits, in place."""
    _dev_or_pinned(target_logits, "target_logits", torch.float32)
    B, n, V = target_logits.shape
    R = n
    Vd = V
    if draft_logits is not None:
        _dev(draft_logits, "draft_logits", torch.float32)
        R = draft_logits.shape[1]
        Vd = draft_logits.shape[2]
    _dev(tokens, "tokens", torch.int32)
    _dev(parent, "parent", torch.int32)
    if draft_row is not None:
        _dev(draft_row, "draft_row", torch.int32)
    dev = tokens.device
    D = int(max_depth)
    accept_len = torch.empty(B, dtype=torch.int32, device=dev) if accept_len is None else accept_len
    path = torch.empty(B, D + 1, dtype=torch.int32, device=dev) if path is None else path
    emit = torch.empty(B, D + 1, dtype=torch.int32, device=dev) if emit is None else emit
    if row_stats is not None:
        _dev(row_stats, "row_stats", torch.float32)
    if (top_k or top_p) and temperature > 0:
        if t2d is not None:
            raise ValueError("top-k / top-p filtering with a draft vocabulary is not offered")
        need = int(lib().eagle_verify_filter_workspace_size(B, n, R))
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        _dev(workspace, "workspace")
        _check("eagle_verify_accept_filtered", lib().eagle_verify_accept_filtered(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_row), _ptr(tokens), _ptr(parent),
            B, n, V, R, D, float(temperature), int(seed) & (2**64 - 1), int(top_k), float(top_p),
            _ptr(accept_len), _ptr(path), _ptr(emit), _ptr(row_stats), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(_status(dev_status, dev)),
            _stream(stream)))
        return accept_len, path, emit
    if t2d is not None:
        _dev(t2d, "t2d", torch.int32)
        _check("eagle_verify_accept_d2t", lib().eagle_verify_accept_d2t(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_row), _ptr(tokens), _ptr(parent),
            B, n, V, R, Vd, _ptr(t2d), D, float(temperature), int(seed) & (2**64 - 1),
            _ptr(accept_len), _ptr(path), _ptr(emit), _ptr(row_stats),
            _ptr(_status(dev_status, dev)), _stream(stream)))
        return accept_len, path, emit
    if draft_logits is not None and Vd != V:
        raise ValueError("draft rows over another vocabulary need t2d")
    _check("eagle_verify_accept", lib().eagle_verify_accept(
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_row), _ptr(tokens), _ptr(parent),
        B, n, V, R, D, float(temperature), int(seed) & (2**64 - 1),
        _ptr(accept_len), _ptr(path), _ptr(emit), _ptr(row_stats),
        _ptr(_status(dev_status, dev)), _stream(stream)))
    return accept_len, path, emit


def eagle_verify_accept_sharded(target_shards, draft_shards, shard_begin, tokens, parent, max_depth,
                                temperature, seed, draft_row=None, accept_len=None, path=None,
                                emit=None, row_stats=None, dev_status=None, stream=None):
    """Vocab-parallel verify: shard r of every target row ([B, n, Vr]) and draft row
    ([B, R, Vr]) holds the ids shard_begin[r] .. shard_begin[r+1]-1 (shard_begin: S + 1
    ints, 0 first, V last).  Returns (accept_len, path, emit) as eagle_verify_accept."""
    S = len(target_shards)
    begin = [int(x) for x in shard_begin]
    if len(begin) != S + 1:
        raise ValueError("shard_begin needs one entry per shard plus the vocabulary size")
    for r, t in enumerate(target_shards):
        _dev(t, f"target_shards[{r}]", torch.float32)
        if t.shape[-1] != begin[r + 1] - begin[r]:
            raise ValueError(f"target_shards[{r}] does not hold ids {begin[r]}..{begin[r + 1] - 1}")
    B, n = target_shards[0].shape[:2]
    V = begin[-1]
    R = n
    dptrs = None
    if draft_shards is not None:
        if len(draft_shards) != S:
            raise ValueError("one draft shard per target shard")
        for r, t in enumerate(draft_shards):
            _dev(t, f"draft_shards[{r}]", torch.float32)
        R = draft_shards[0].shape[1]
        dptrs = (ctypes.c_void_p * S)(*[t.data_ptr() for t in draft_shards])
    tptrs = (ctypes.c_void_p * S)(*[t.data_ptr() for t in target_shards])
    cbeg = (ctypes.c_int32 * (S + 1))(*begin)
    _dev(tokens, "tokens", torch.int32)
    _dev(parent, "parent", torch.int32)
    if draft_row is not None:
        _dev(draft_row, "draft_row", torch.int32)
    dev = tokens.device
    D = int(max_depth)
    accept_len = torch.empty(B, dtype=torch.int32, device=dev) if accept_len is None else accept_len
    path = torch.empty(B, D + 1, dtype=torch.int32, device=dev) if path is None else path
    emit = torch.empty(B, D + 1, dtype=torch.int32, device=dev) if emit is None else emit
    if row_stats is not None:
        _dev(row_stats, "row_stats", torch.float32)
    _check("eagle_verify_accept_sharded", lib().eagle_verify_accept_sharded(
        tptrs, dptrs, cbeg, S, _ptr(draft_row), _ptr(tokens), _ptr(parent), B, n, V, R, D,
        float(temperature), int(seed) & (2**64 - 1), _ptr(accept_len), _ptr(path), _ptr(emit),
        _ptr(row_stats), _ptr(_status(dev_status, dev)), _stream(stream)))
    return accept_len, path, emit


def eagle_kv_compact(k_cache, v_cache, kv_len, path, accept_len, max_depth, dev_status=None,
                     stream=None):
    """k/v cache [n_layers,B,Hkv,Lmax,d] bf16 (in place); kv_len updated in place."""
    _dev(k_cache, "k_cache", torch.bfloat16)
    _dev(v_cache, "v_cache", torch.bfloat16)
    _dev(kv_len, "kv_len", torch.int32)
    _dev(path, "path", torch.int32)
    _dev(accept_len, "accept_len", torch.int32)
    nl, B, Hkv, Lmax, d = k_cache.shape
    _check("eagle_kv_compact", lib().eagle_kv_compact(
        _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(path), _ptr(accept_len),
        nl, B, Hkv, d, Lmax, int(max_depth), _ptr(_status(dev_status, k_cache.device)),
        _stream(stream)))


def expand_scratch_size(B, V, top_k) -> int:
    return int(lib().eagle2_expand_scratch_size(B, V, top_k))


def eagle2_expand(level, final, logits, top_k, depth, n_out, tree_state, hidden=None,
                  lm_head_w=None, out_tokens=None, out_parent=None, out_draft_row=None,
                  frontier_tokens=None, dev_status=None, stream=None, partials=None, d2t=None):
    """One EAGLE-2 level over draft-logit storage logits [B, R, V] (f32).  With a
    partials buffer the level's statistics come from the GEMM epilogue's per-tile
    partials (written by this call's GEMM when hidden is given, else by a prior
    eagle_lmhead_gemm(..., partials=...) for the level's rows) and its top-k from a
    rescan of the few tiles that can hold it.  With d2t (int32 [V]) V is a draft
    vocabulary and the tokens written are target ids d + d2t[d]."""
    _dev(logits, "logits", torch.float32)
    _dev(tree_state, "tree_state")
    B, R, V = logits.shape
    H = 0
    if hidden is not None:
        _dev(hidden, "hidden", torch.bfloat16)
        _dev(lm_head_w, "lm_head_w", torch.bfloat16)
        H = hidden.shape[-1]
    for name, t in (("out_tokens", out_tokens), ("out_parent", out_parent),
                    ("out_draft_row", out_draft_row), ("frontier_tokens", frontier_tokens)):
        if t is not None:
            _dev(t, name, torch.int32)
    nbytes = tree_state.numel() * tree_state.element_size()
    sbytes = 0
    if partials is not None:
        _dev(partials, "partials", torch.float32)
        sbytes = partials.numel() * partials.element_size()
    if d2t is not None:
        _dev(d2t, "d2t", torch.int32)
        if d2t.numel() != V:
            raise ValueError("d2t needs one entry per draft id")
        _check("eagle2_expand_d2t", lib().eagle2_expand_d2t(
            int(level), int(final), _ptr(hidden), _ptr(lm_head_w), _ptr(logits), B, H, V, top_k,
            depth, n_out, _ptr(tree_state), nbytes, _ptr(partials), sbytes, _ptr(d2t),
            _ptr(out_tokens), _ptr(out_parent), _ptr(out_draft_row), _ptr(frontier_tokens),
            _ptr(_status(dev_status, logits.device)), _stream(stream)))
        return
    _check("eagle2_expand", lib().eagle2_expand(
        int(level), int(final), _ptr(hidden), _ptr(lm_head_w), _ptr(logits), B, H, V, top_k, depth,
        n_out, _ptr(tree_state), nbytes, _ptr(partials), sbytes, _ptr(out_tokens), _ptr(out_parent),
        _ptr(out_draft_row), _ptr(frontier_tokens), _ptr(_status(dev_status, logits.device)),
        _stream(stream)))


def eagle2_tree_candidates(tree_state, B, top_k, depth, stream=None):
    """Every candidate of a tree state as CUDA tensors [B, C]: dict(value, conf (f32),
    token, parent, depth, draft_row (int32)), C = 1 + top_k + (depth - 1) * top_k^2."""
    _dev(tree_state, "tree_state")
    C = 1 + top_k + (depth - 1) * top_k * top_k
    dev = tree_state.device
    out = {"value": torch.empty(B, C, device=dev), "conf": torch.empty(B, C, device=dev)}
    for name in ("token", "parent", "depth", "draft_row"):
        out[name] = torch.empty(B, C, dtype=torch.int32, device=dev)
    nbytes = tree_state.numel() * tree_state.element_size()
    _check("eagle2_tree_candidates", lib().eagle2_tree_candidates(
        _ptr(tree_state), nbytes, B, top_k, depth, _ptr(out["value"]), _ptr(out["conf"]),
        _ptr(out["token"]), _ptr(out["parent"]), _ptr(out["depth"]), _ptr(out["draft_row"]),
        _stream(stream)))
    return out


def eagle_static_tree(choices):
    """Plan a static draft tree from its choices (rank paths from the root) on the host.
    Returns dict(parent, rank, depth, draft_row) of int32 numpy arrays [n]."""
    import numpy as np
    n_choices = len(choices)
    max_len = max((len(c) for c in choices), default=1)
    ranks = np.zeros((max(n_choices, 1), max_len), np.int32)
    lens = np.zeros(max(n_choices, 1), np.int32)
    for i, c in enumerate(choices):
        ranks[i, :len(c)] = c
        lens[i] = len(c)
    n_max = n_choices + 1
    out = {k: np.zeros(n_max, np.int32) for k in ("parent", "rank", "depth", "draft_row")}
    n_nodes = np.zeros(1, np.int32)
    adr = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    _check("eagle_static_tree", lib().eagle_static_tree(
        adr(ranks), adr(lens), n_choices, max_len, n_max, adr(out["parent"]), adr(out["rank"]),
        adr(out["depth"]), adr(out["draft_row"]), adr(n_nodes)))
    n = int(n_nodes[0])
    return {k: v[:n] for k, v in out.items()}


def eagle_static_tree_level(level, logits, parent, rank, depth, draft_row, tokens,
                            dev_status=None, stream=None):
    """Tokens of the nodes at depth `level` of a static tree (device int32 arrays [n]),
    from the internal nodes' draft rows logits [B, R, V] (f32), into tokens [B, n]."""
    _dev(logits, "logits", torch.float32)
    for name, t in (("parent", parent), ("rank", rank), ("depth", depth),
                    ("draft_row", draft_row), ("tokens", tokens)):
        _dev(t, name, torch.int32)
    B, R, V = logits.shape
    _check("eagle_static_tree_level", lib().eagle_static_tree_level(
        int(level), _ptr(logits), _ptr(parent), _ptr(rank), _ptr(depth), _ptr(draft_row),
        parent.numel(), B, R, V, _ptr(tokens), _ptr(_status(dev_status, logits.device)),
        _stream(stream)))


def eagle2_expand_static_state(level, final, logits, top_k, depth, n_out, hidden=None,
                               lm_head_w=None, out_tokens=None, out_parent=None,
                               out_draft_row=None, frontier_tokens=None, dev_status=None,
                               stream=None):
    """eagle2_expand with the tree state kept in the library's own fixed device array
    (no scratch argument; one tree at a time per device, levels in order)."""
    _dev(logits, "logits", torch.float32)
    B, R, V = logits.shape
    H = 0
    if hidden is not None:
        _dev(hidden, "hidden", torch.bfloat16)
        _dev(lm_head_w, "lm_head_w", torch.bfloat16)
        H = hidden.shape[-1]
    for name, t in (("out_tokens", out_tokens), ("out_parent", out_parent),
                    ("out_draft_row", out_draft_row), ("frontier_tokens", frontier_tokens)):
        if t is not None:
            _dev(t, name, torch.int32)
    _check("eagle2_expand_static_state", lib().eagle2_expand_static_state(
        int(level), int(final), _ptr(hidden), _ptr(lm_head_w), _ptr(logits), B, H, V, top_k,
        depth, n_out, _ptr(out_tokens), _ptr(out_parent), _ptr(out_draft_row),
        _ptr(frontier_tokens), _ptr(_status(dev_status, logits.device)), _stream(stream)))


def eagle_softmax_stats(logits, temperature, row_max=None, row_sum=None, row_argmax=None,
                        dev_status=None, stream=None, argmax=True):
    """(row_max, row_sum, row_argmax) of softmax(logits / T) per row.  At T > 0 the
    argmax is computed only when `argmax` is true (or row_argmax is given); it is
    returned as None otherwise."""
    _dev(logits, "logits", torch.float32)
    V = logits.shape[-1]
    rows = logits.numel() // V
    dev = logits.device
    shp = logits.shape[:-1]
    if temperature > 0:
        row_max = torch.empty(shp, dtype=torch.float32, device=dev) if row_max is None else row_max
        row_sum = torch.empty(shp, dtype=torch.float32, device=dev) if row_sum is None else row_sum
    if row_argmax is None and (argmax or temperature <= 0):
        row_argmax = torch.empty(shp, dtype=torch.int32, device=dev)
    _check("eagle_softmax_stats", lib().eagle_softmax_stats(
        _ptr(logits), rows, V, float(temperature), _ptr(row_max), _ptr(row_sum), _ptr(row_argmax),
        _ptr(_status(dev_status, dev)), _stream(stream)))
    return row_max, row_sum, row_argmax


def eagle_lmhead_gemm(hidden, w, out=None, ldo=None, rows_per_group=None, group_stride=0,
                      row_offset=0, dev_status=None, stream=None, partials=None):
    """out[row(m)] = hidden[m] . W^T, hidden [M,K], w [N,K] bf16, out f32.  With a
    partials buffer [M, ceil(N/256), 2] (f32) also each row's per-tile (max, sum of
    exponentials)."""
    _dev(hidden, "hidden", torch.bfloat16)
    _dev(w, "w", torch.bfloat16)
    M, K = hidden.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=hidden.device)
    _dev(out, "out", torch.float32)
    ldo = N if ldo is None else ldo
    rpg = M if rows_per_group is None else rows_per_group
    if partials is not None:
        _dev(partials, "partials", torch.float32)
    _check("eagle_lmhead_gemm", lib().eagle_lmhead_gemm(
        _ptr(hidden), _ptr(w), _ptr(out), M, K, N, int(ldo), int(rpg), int(group_stride),
        int(row_offset), _ptr(partials), _ptr(_status(dev_status, hidden.device)),
        _stream(stream)))
    return out
