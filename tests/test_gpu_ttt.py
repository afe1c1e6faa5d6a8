"""GPU parity of eagle_ttt_attn (training-time-test attention) against the
double-precision oracle.

Tolerance: per (sequence, position, head) row, max|O_gpu - O_ref| / max|O_ref| <= 1e-2,
as for the tree attention (bf16 inputs and output, fp32 accumulation, P rounded to
bf16 for the PV product, the diagonal keys included).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import attn_row_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2
D = 128


def _run(q, k, v, r, scale):
    import eagle_tree_speculative_gb300 as E
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = E.eagle_ttt_attn(q.cuda(), k.cuda(), v.cuda(), r, scale=scale, dev_status=st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(st.item())


@pytest.mark.parametrize("B,S,Hq,Hkv,R1,r", [
    (2, 300, 32, 8, 4, 0),      # causal only; 1200 rows = 9 full tiles + 48, keys span 3 tiles
    (2, 300, 32, 8, 4, 3),      # deepest stored round
    (1, 130, 4, 4, 3, 2),       # G = 1: one position per row, a 2-key ragged key tail
    (1, 200, 64, 8, 8, 5),      # G = 8
    (2, 100, 6, 2, 5, 1),       # G = 3: positions straddle row tiles
    (1, 1, 8, 2, 2, 1),         # a single position
    (1, 129, 8, 8, 16, 15),     # the most rounds: 15 diagonal boxes of one round each
    (2, 160, 32, 8, 16, 13),    # G = 4: 4 diagonal boxes of 4 rounds, stages reused
])
def test_matches_oracle(B, S, Hq, Hkv, R1, r):
    q, k, v = W.ttt_inputs(B, S, Hq, Hkv, D, R1, seed=31 + r)
    scale = D ** -0.5
    got, st = _run(q, k, v, r, scale)
    assert st == 0
    ref = oracle.ttt_attn(q, k, v, r, scale)
    err = attn_row_rel_err(got, ref)
    assert err.max() <= TOL, (err.max(), np.unravel_index(err.argmax(), err.shape))


@pytest.mark.parametrize("Hq,Hkv,R1,r", [(32, 8, 8, 3), (6, 2, 6, 2), (8, 8, 5, 1)])
def test_rounds_after_r_are_never_read(Hq, Hkv, R1, r):
    """Rounds r+1 .. R1-1 hold NaN and +inf (not yet simulated); the output must match
    the oracle, which reads only rounds 0 .. r.  The diagonal boxes cover more rounds
    than r needs (G = 4: 4 rounds per box, G = 3: 2, G = 1: 1)."""
    B, S = 2, 150
    q, k, v = W.ttt_inputs(B, S, Hq, Hkv, D, R1, seed=57 + r)
    k, v = k.clone(), v.clone()
    k[:, :, r + 1:] = float("nan")
    v[:, :, r + 1:] = float("nan")
    v[:, :, r + 1:, ::3] = float("inf")
    scale = D ** -0.5
    got, st = _run(q, k, v, r, scale)
    assert st == 0
    assert np.isfinite(got).all()
    ref = oracle.ttt_attn(q, k, v, r, scale)
    assert attn_row_rel_err(got, ref).max() <= TOL


def test_full_size_rows_sampled():
    """8 sequences x 2048 positions, Llama-3-8B heads (32 q / 8 kv), round 7 of 8: the
    benchmark's shape.  A row at position i depends only on positions 0..i, so the
    oracle recomputes sampled rows from the prefix of one (sequence, kv head) group."""
    B, S, Hq, Hkv, R1, r = 8, 2048, 32, 8, 8, 7
    G = Hq // Hkv
    q, k, v = W.ttt_inputs(B, S, Hq, Hkv, D, R1, seed=41)
    scale = D ** -0.5
    got, st = _run(q, k, v, r, scale)
    assert st == 0
    for b, kvh, i in [(0, 0, 0), (3, 5, 127), (5, 2, 1000), (7, 7, S - 1)]:
        qs = q[b:b + 1, :i + 1, kvh * G:(kvh + 1) * G].contiguous()
        ks = k[b:b + 1, kvh:kvh + 1, :, :i + 1].contiguous()
        vs = v[b:b + 1, kvh:kvh + 1, :, :i + 1].contiguous()
        ref = oracle.ttt_attn(qs, ks, vs, r, scale)[0, i]
        err = attn_row_rel_err(got[b, i, kvh * G:(kvh + 1) * G], ref)
        assert err.max() <= TOL, (b, kvh, i, err.max())


def test_empty_batch_and_argument_errors():
    import eagle_tree_speculative_gb300 as E
    q, k, v = W.ttt_inputs(1, 8, 4, 2, D, 3, seed=5)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    out = E.eagle_ttt_attn(q[:0], k[:0], v[:0], 1)
    assert out.shape[0] == 0
    for r in (-1, 3):
        with pytest.raises(RuntimeError):
            E.eagle_ttt_attn(q, k, v, r)
    k17 = torch.zeros(1, 2, 17, 8, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        E.eagle_ttt_attn(q, k17, k17.clone(), 1)
