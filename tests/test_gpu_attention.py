"""GPU parity of eagle_tree_attn against the double-precision oracle.

Tolerance: per (sequence, node, head) row, max|O_gpu - O_ref| / max|O_ref| <= 1e-2
(bf16 inputs and output, fp32 accumulation, P rounded to bf16 for the PV product).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import attn_row_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _run(q, k, v, kv_len, parent, scale, status=None):
    import eagle_tree_speculative_gb300 as E
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    out = E.eagle_tree_attn(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(kv_len).cuda(),
                            torch.from_numpy(np.ascontiguousarray(parent)).cuda(), scale=scale,
                            dev_status=st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(st.item())


def _check(B, n, Hq, Hkv, kv_len, Lmax, seed, parent=None, sample=None):
    d = 128
    q, k, v, kv_len = W.attn_inputs(B, n, Hq, Hkv, d, kv_len, Lmax, seed)
    if parent is None:
        parent = np.stack([W.random_tree(n, 8, seed, b) for b in range(B)])
    scale = d ** -0.5
    got, st = _run(q, k, v, kv_len, parent, scale)
    assert st == 0
    bs = range(B) if sample is None else sample
    for b in bs:
        ref = oracle.tree_attn(q[b:b + 1], k[b:b + 1], v[b:b + 1], kv_len[b:b + 1],
                               parent[b:b + 1], scale)
        err = attn_row_rel_err(got[b:b + 1], ref)
        assert err.max() <= TOL, (b, err.max())
    return got


def test_small_ragged_lengths_several_tiles():
    _check(B=3, n=13, Hq=8, Hkv=2, kv_len=[0, 37, 200], Lmax=230, seed=1)


def test_gqa_groups_and_row_blocks():
    # n * G = 21 * 8 = 168 rows: two 128-row blocks, ragged tail
    _check(B=2, n=21, Hq=16, Hkv=2, kv_len=[300, 129], Lmax=330, seed=2)


def test_lone_root_with_empty_cache_returns_value_row():
    q, k, v, kv_len = W.attn_inputs(2, 1, 4, 2, 128, 0, 8, seed=3)
    got, st = _run(q, k, v, kv_len, np.full((2, 1), -1, np.int32), 0.1)
    assert st == 0
    for b in range(2):
        for h in range(4):
            np.testing.assert_array_equal(got[b, 0, h], v[b, h // 2, 0].float().numpy())


def test_chain_tree_matches_oracle_causal_case():
    _check(B=2, n=20, Hq=4, Hkv=4, kv_len=[64, 100], Lmax=128, seed=4,
           parent=np.stack([W.chain_tree(20)] * 2))


def test_vicuna13b_shape_b1_split_kv():
    """B=1, 60 nodes, 40 heads, L=2048: the split-KV path; every row checked."""
    cfg = W.CONFIGS["eagle2_b1"]
    _check(B=1, n=cfg.n, Hq=cfg.Hq, Hkv=cfg.Hkv, kv_len=cfg.L, Lmax=cfg.Lmax, seed=5)


def test_llama3_8b_shape_b64_full_size_sampled():
    """B=64, 60 nodes, 32/8 heads, L=4096 (the benchmark launch); 3 sequences checked."""
    cfg = W.CONFIGS["eagle3_b64"]
    _check(B=cfg.B, n=cfg.n, Hq=cfg.Hq, Hkv=cfg.Hkv, kv_len=cfg.L, Lmax=cfg.Lmax, seed=6,
           sample=[0, 31, 63])


@pytest.mark.parametrize("B,L,sample", [
    (1, 8192, None), (1, 16384, None), (1, 32768, None),          # every row; split KV
    (8, 512, [0, 7]), (8, 16384, [0, 7]), (8, 32768, [5]),
    (32, 2048, [0, 31]), (32, 16384, [17]),
    (64, 1024, [0, 63]), (64, 4096, [0, 40, 63]), (64, 8192, [63])])
def test_llama70b_shape_sweep_points(B, L, sample):
    """The Llama-70B sweep's attention (64 q / 8 kv heads, 48-node trees) over its batch
    sizes and KV lengths up to 32768; sampled sequences are checked row by row."""
    cfg = W.CONFIGS["sweep_70b"]
    _check(B=B, n=cfg.n, Hq=cfg.Hq, Hkv=cfg.Hkv, kv_len=L, Lmax=L + cfg.n, seed=7 + B + L,
           sample=sample)


@pytest.mark.parametrize("B,n,Hq,Hkv,L", [
    (1, 60, 32, 8, [8192]),            # two M-tiles, keys split across CTAs
    (2, 40, 16, 4, [1000, 77]),        # 160 rows: a part-empty second M-tile;
                                       # 77 + 40 keys fit in less than one key tile
    (2, 60, 64, 8, [500, 2000]),       # 480 rows: four M-tiles per (sequence, kv head)
    (3, 33, 32, 4, [129, 1, 4096]),    # 264 rows: three M-tiles, one holding 8 rows
])
def test_row_tiles_of_every_count(B, n, Hq, Hkv, L):
    """(node, head) rows of one (sequence, kv head) in one to four 128-row M-tiles, with
    ragged last tiles and caches shorter than one key tile.  Every row checked."""
    _check(B=B, n=n, Hq=Hq, Hkv=Hkv, kv_len=L, Lmax=max(L) + n, seed=31 + n)


def test_capacity_and_tree_errors_set_status_and_zero_output():
    import eagle_tree_speculative_gb300 as E
    q, k, v, kv_len = W.attn_inputs(2, 4, 2, 1, 128, [10, 3], 13, seed=8)
    parent = np.array([[-1, 0, 1, 2], [-1, 2, 0, 1]], np.int32)     # second tree invalid
    got, st = _run(q, k, v, kv_len, parent, 0.1)
    assert st & E.EAGLE_DEV_CAPACITY and st & E.EAGLE_DEV_BAD_TREE   # 10 + 4 > 13 in seq 0
    assert np.all(got == 0)


@pytest.mark.parametrize("Hq,Hkv,n,L,Lmax", [(32, 8, 60, [200, 77, 333], 512),
                                             (8, 8, 13, [200, 77, 333], 512),
                                             (32, 8, 30, [1000], 2048)])
def test_unwritten_cache_rows_past_the_tree_do_not_leak(Hq, Hkv, n, L, Lmax):
    """Cache rows at and beyond L + n are not part of the attention; a cache that was
    never written there may hold anything.  Those rows are set to NaN and +inf here (K
    and V); the output must still match the oracle, which never reads them.  The last
    key tile is partial in every case; 77 + 13 keys fit in less than one tile; one
    sequence at 2048 rows splits its keys across CTAs."""
    B, d = len(L), 128
    q, k, v, kv_len = W.attn_inputs(B, n, Hq, Hkv, d, L, Lmax, seed=21)
    k, v = k.clone(), v.clone()
    for b in range(B):
        k[b, :, L[b] + n:] = float("nan")
        v[b, :, L[b] + n:] = float("nan")
        v[b, :, L[b] + n + 1::3] = float("inf")
    parent = np.stack([W.random_tree(n, 6, 21, b) for b in range(B)])
    scale = d ** -0.5
    got, st = _run(q, k, v, kv_len, parent, scale)
    assert st == 0
    assert np.isfinite(got).all()
    for b in range(B):
        ref = oracle.tree_attn(q[b:b + 1], k[b:b + 1], v[b:b + 1], kv_len[b:b + 1],
                               parent[b:b + 1], scale)
        assert attn_row_rel_err(got[b:b + 1], ref).max() <= TOL
