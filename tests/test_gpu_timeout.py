"""Failure detection without a fault: an expired bounded wait reports a status.

eagle_wait_selftest waits on an mbarrier that nothing completes, with the same
polling loop as the pipelined kernels, for a short limit; it must set
EAGLE_DEV_TIMEOUT and return, and the context must stay usable."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def test_expired_wait_sets_timeout_status_and_context_survives():
    import eagle_tree_speculative_gb300 as E
    L = E.lib()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.eagle_wait_selftest(st.data_ptr(), 2_000_000, stream) == 0     # ~1 ms
    torch.cuda.synchronize()
    assert int(st.item()) == E.EAGLE_DEV_TIMEOUT
    # out-of-range limits are rejected on the host
    assert L.eagle_wait_selftest(st.data_ptr(), 0, stream) == 1
    assert L.eagle_wait_selftest(None, 10, stream) == 1
    # the next real call runs normally
    V, n = 512, 4
    tgt = W.per_seq_normal(2, (n, V), 1.0, 3, W.TAG_TARGET)
    par = np.tile(W.chain_tree(n), (2, 1))
    tok = np.tile(np.array([-1, 1, 2, 3], np.int32), (2, 1))
    st.zero_()
    acc, path, emit = E.eagle_verify_accept(
        torch.from_numpy(tgt).cuda(), None, torch.from_numpy(tok).cuda(),
        torch.from_numpy(par).cuda(), 3, 0.0, 0, dev_status=st)
    torch.cuda.synchronize()
    ref = oracle.verify_accept(tgt, tgt, tok, par, 3, 0.0, 0)
    assert int(st.item()) == 0
    assert np.array_equal(acc.cpu().numpy(), ref["accept_len"])
