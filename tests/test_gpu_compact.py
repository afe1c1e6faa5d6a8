"""GPU parity of eagle_kv_compact: bit-exact against the oracle's literal copy."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).copy()


def _run(k, v, kv_len, path, acc, D):
    import eagle_tree_speculative_gb300 as E
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kg, vg = k.cuda(), v.cuda()
    kl = torch.from_numpy(kv_len.copy()).cuda()
    E.eagle_kv_compact(kg, vg, kl, torch.from_numpy(path).cuda(), torch.from_numpy(acc).cuda(), D,
                       dev_status=st)
    torch.cuda.synchronize()
    return _bits(kg), _bits(vg), kl.cpu().numpy(), int(st.item())


def test_overlapping_paths_and_skips_match_oracle():
    nl, B, H, d, Lmax, D = 3, 5, 2, 128, 40, 6
    k, v = W.kv_cache(nl, B, H, Lmax, d, seed=1)
    kv_len = np.array([4, 0, 9, 20, 3], np.int32)
    path = np.full((B, D + 1), -1, np.int32)
    path[0, :3] = [0, 2, 7]                 # row 2 is both a source and a destination
    path[1, :5] = [0, 1, 3, 4, 9]
    path[2, :1] = [0]
    path[3, :7] = [0, 1, 2, 3, 4, 5, 6]     # all in place
    path[4, :3] = [0, 5, 6]
    acc = np.array([2, 4, 0, 6, -1], np.int32)  # last sequence failed verification
    kr, vr = _bits(k), _bits(v)
    klr = kv_len.copy()
    assert oracle.kv_compact(kr, vr, klr, path, acc, D) == 0
    kg, vg, klg, st = _run(k, v, kv_len, path, acc, D)
    assert st == 0
    assert np.array_equal(klg, klr)
    assert np.array_equal(kg, kr) and np.array_equal(vg, vr)


def test_two_sequence_rollback_exercise():
    nl, B, H, d, Lmax, D = 2, 2, 2, 128, 24, 4
    k, v = W.kv_cache(nl, B, H, Lmax, d, seed=2)
    kv_len = np.array([10, 7], np.int32)
    path = np.array([[0, 1, 2, 3, 4], [0, 1, -1, -1, -1]], np.int32)
    kg, vg, klg, st = _run(k, v, kv_len, path, np.array([4, 1], np.int32), D)
    assert st == 0 and list(klg) == [15, 9]
    assert np.array_equal(kg, _bits(k)) and np.array_equal(vg, _bits(v))


def test_capacity_and_bad_path_flagged_and_skipped():
    import eagle_tree_speculative_gb300 as E
    nl, B, H, d, Lmax, D = 1, 2, 1, 128, 12, 3
    k, v = W.kv_cache(nl, B, H, Lmax, d, seed=3)
    kv_len = np.array([9, 2], np.int32)
    path = np.array([[0, 1, 3, -1], [0, 2, 1, -1]], np.int32)  # seq 0 overflows, seq 1 not increasing
    kg, vg, klg, st = _run(k, v, kv_len, path, np.array([2, 2], np.int32), D)
    assert st & E.EAGLE_DEV_CAPACITY and st & E.EAGLE_DEV_BAD_TREE
    assert list(klg) == [9, 2]
    assert np.array_equal(kg, _bits(k)) and np.array_equal(vg, _bits(v))


def test_full_size_32_layers_b64_sampled_slices():
    """Llama-3-8B shape: 32 layers x 64 seqs x 8 kv heads, L=4096 + 60 tree rows.
    The cache is filled by torch's device RNG; sampled (layer, seq, head) slices are
    copied out before and after and compacted by the oracle."""
    nl, B, H, d = 32, 64, 8, 128
    L, n, D = 4096, 60, 8
    Lmax = L + n
    g = torch.Generator(device="cuda").manual_seed(0)
    k = torch.randint(-2**15, 2**15 - 1, (nl, B, H, Lmax, d), dtype=torch.int16, device="cuda",
                      generator=g).view(torch.bfloat16)
    v = torch.randint(-2**15, 2**15 - 1, (nl, B, H, Lmax, d), dtype=torch.int16, device="cuda",
                      generator=g).view(torch.bfloat16)
    rng = W.rng(4, 4)
    acc = rng.integers(0, D + 1, size=B).astype(np.int32)
    path = np.full((B, D + 1), -1, np.int32)
    for b in range(B):
        picks = np.sort(rng.choice(np.arange(1, n), size=acc[b], replace=False))
        path[b, :acc[b] + 1] = np.concatenate([[0], picks])
    kv_len = np.full(B, L, np.int32)
    samples = [(0, 0, 0), (31, 63, 7), (17, 5, 3), (9, 40, 6)]
    before = [(_bits(k[l, b, h]), _bits(v[l, b, h])) for l, b, h in samples]
    import eagle_tree_speculative_gb300 as E
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kl = torch.from_numpy(kv_len).cuda()
    E.eagle_kv_compact(k, v, kl, torch.from_numpy(path).cuda(), torch.from_numpy(acc).cuda(), D,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(kl.cpu().numpy(), kv_len + acc + 1)
    for (l, b, h), (kb, vb) in zip(samples, before):
        kr, vr = kb[None, None, None].copy(), vb[None, None, None].copy()
        klr = kv_len[b:b + 1].copy()
        oracle.kv_compact(kr, vr, klr, path[b:b + 1], acc[b:b + 1], D)
        assert np.array_equal(_bits(k[l, b, h]), kr[0, 0, 0])
        assert np.array_equal(_bits(v[l, b, h]), vr[0, 0, 0])
