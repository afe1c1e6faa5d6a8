"""eagle2_expand_static_state: the tree state lives in the library's own device array.

It serves callers that may not allocate device memory once they run: a serving loop
that reserves its memory at start-up, or code behind another framework's allocator.
Called through the C ABI (ctypes, raw device pointers) and compared bit for bit with
eagle2_expand on caller-provided scratch, for two trees expanded one after the other,
so the second tree runs on whatever the first left in the array; a full tree through
it leaves the device's free memory and torch's allocation unchanged.  This file sorts
last so that the array has also seen every earlier test's process state.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

EAGLE_ERR_CAPACITY = 3


def _L():
    import eagle_tree_speculative_gb300 as E
    return E, E.lib()


def _run_tree(logits, k, D, n_out, static, hidden=None, w=None):
    """All D levels of one tree; returns tokens, parents, draft rows, frontier, status."""
    E, L = _L()
    B, R, V = logits.shape
    H = 0 if hidden is None else hidden[0].shape[-1]
    dev = logits.device
    tok = torch.full((B, n_out), -5, dtype=torch.int32, device=dev)
    par = torch.full_like(tok, -5)
    row = torch.full_like(tok, -5)
    fr = torch.full((B, k), -5, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    state = None
    if not static:
        state = torch.empty(int(L.eagle2_tree_state_size(B, k, D)), dtype=torch.uint8, device=dev)
    for lvl in range(1, D + 1):
        hp = None if hidden is None else hidden[lvl - 1].data_ptr()
        wp = None if w is None else w.data_ptr()
        common_head = (lvl, int(lvl == D), hp, wp, logits.data_ptr(), B, H, V, k, D, n_out)
        common_tail = (tok.data_ptr(), par.data_ptr(), row.data_ptr(), fr.data_ptr(),
                       st.data_ptr(), stream)
        if static:
            rc = L.eagle2_expand_static_state(*common_head, *common_tail)
        else:
            rc = L.eagle2_expand(*common_head, state.data_ptr(), state.numel(), None, 0, *common_tail)
        assert rc == 0, E.lib().eagle_status_str(rc)
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), par.cpu().numpy(), row.cpu().numpy(), fr.cpu().numpy(),
            int(st.item()))


def _logits(seed, B, V):
    cfg = W.CONFIGS["expand_b64"]
    _, drows = W.tree_draft_rows(cfg, seed=seed, B=B, V=V)
    return torch.from_numpy(drows).cuda()


def test_static_state_matches_scratch_entry_on_two_trees_in_a_row():
    cfg = W.CONFIGS["expand_b64"]          # top-10, depth 8, 60 nodes
    k, D, n = cfg.top_k, cfg.depth, cfg.n
    trees = [_logits(21, 64, 32000), _logits(22, 64, 32000)]
    for lg in trees:
        got = _run_tree(lg, k, D, n, static=True)
        ref = _run_tree(lg, k, D, n, static=False)
        assert got[4] == 0 and ref[4] == 0
        for g, r in zip(got[:4], ref[:4]):
            assert np.array_equal(g, r)
        assert (got[0][:, 1:] >= 0).all() and (got[1][:, 0] == -1).all()


def test_static_state_fed_by_gemm_then_smaller_tree():
    """A GEMM-fed tree (hidden -> tcgen05 LM head -> expansion), then a smaller tree
    with other k / depth on the same array: both equal the scratch entry's result."""
    B, k, D, n_out, H, V = 4, 10, 4, 30, 4096, 8192
    R = 1 + (D - 1) * k
    w = W.lm_head(V, H, 0.02, 23, block=1024).cuda()
    hid = [W.hidden_states(B, 1 if l == 1 else k, H, l, 23).cuda() for l in range(1, D + 1)]
    lg_s = torch.zeros(B, R, V, device="cuda")
    lg_r = torch.zeros(B, R, V, device="cuda")
    got = _run_tree(lg_s, k, D, n_out, static=True, hidden=hid, w=w)
    ref = _run_tree(lg_r, k, D, n_out, static=False, hidden=hid, w=w)
    assert got[4] == 0 and ref[4] == 0
    for g, r in zip(got[:4], ref[:4]):
        assert np.array_equal(g, r)
    assert torch.equal(lg_s, lg_r)

    small = _logits(24, 7, 3000)[:, :1 + 2 * 4]      # k = 4, depth 3: R = 9
    small = small.contiguous()
    got = _run_tree(small, 4, 3, 12, static=True)
    ref = _run_tree(small, 4, 3, 12, static=False)
    assert got[4] == 0 and ref[4] == 0
    for g, r in zip(got[:4], ref[:4]):
        assert np.array_equal(g, r)


def test_static_state_rejects_trees_beyond_its_capacity():
    E, L = _L()
    k, D = 10, 8
    per_seq = int(L.eagle2_tree_state_size(1, k, D))
    B = (4 << 20) // per_seq + 1                       # one sequence too many
    assert int(L.eagle2_tree_state_size(B, k, D)) > (4 << 20)
    lg = torch.zeros(B, 1 + (D - 1) * k, 16, device="cuda")
    tok = torch.empty(B, 60, dtype=torch.int32, device="cuda")
    rc = L.eagle2_expand_static_state(1, 0, None, None, lg.data_ptr(), B, 0, 16, k, D, 60,
                                      tok.data_ptr(), None, None, None, None,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == EAGLE_ERR_CAPACITY
    B_ok = (4 << 20) // per_seq
    assert int(L.eagle2_tree_state_size(B_ok, k, D)) <= (4 << 20)


def test_static_state_allocates_nothing():
    """After one warm-up tree (which loads the kernels), a full tree through the
    fixed-array entry point changes neither the device's free memory (cudaMemGetInfo)
    nor torch's allocated bytes."""
    cfg = W.CONFIGS["expand_b64"]
    k, D, n = cfg.top_k, cfg.depth, cfg.n
    lg = _logits(25, 64, 32000)
    B = lg.shape[0]
    E, L = _L()
    dev = lg.device
    tok = torch.empty((B, n), dtype=torch.int32, device=dev)
    par, row = torch.empty_like(tok), torch.empty_like(tok)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def tree():
        for lvl in range(1, D + 1):
            rc = L.eagle2_expand_static_state(lvl, int(lvl == D), None, None, lg.data_ptr(), B, 0,
                                              lg.shape[2], k, D, n, tok.data_ptr(), par.data_ptr(),
                                              row.data_ptr(), None, st.data_ptr(), stream)
            assert rc == 0
        torch.cuda.synchronize()

    tree()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    tree()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, (free0, free1)
    assert int(st.item()) == 0
