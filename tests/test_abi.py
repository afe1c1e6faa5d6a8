"""The C-ABI library builds, loads without a GPU and exports every symbol
include/eagle.h declares; the Python binding declares each of them.  No compute
call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eagle.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle\w*)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    from eagle_tree_speculative_gb300 import build
    import shutil
    if not os.path.exists(build.LIB):
        if shutil.which(build.NVCC) is None:
            pytest.skip("nvcc not available to build the library")
        build.build()
    return build.LIB


def test_header_declares_the_four_calls():
    names = _declared()
    for fn in ("eagle_tree_attn", "eagle_verify_accept", "eagle_kv_compact", "eagle2_expand"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib_path):
    L = ctypes.CDLL(lib_path)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_declares_every_symbol():
    from eagle_tree_speculative_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == _declared()


def test_host_only_queries(lib_path):
    import eagle_tree_speculative_gb300 as E
    assert E.lib().eagle_abi_version() == 100
    assert E.lib().eagle_status_str(2) == b"EAGLE_ERR_SHAPE"
    # workspace and tree-state sizes are pure host arithmetic
    # header, 6 words per candidate (711 at k=10, D=8), frontier, and per (row, segment)
    # of up to 4 vocabulary segments: 3 statistics words + k values + k tokens
    assert E.tree_state_size(64, 10, 8) == 64 * 4 * (4 + 6 * 711 + 16 + 10 * 4 * (3 + 2 * 10))
    assert E.tree_state_size(1, 17, 8) == 0                # top_k above the limit
    assert E.tree_attn_workspace_size(64, 60, 32, 8, 128, 4156) >= 0
    assert E.tree_attn_workspace_size(1, 60, 32, 8, 64, 4156) == 0    # head_dim != 128


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from eagle_tree_speculative_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(_lib.LibraryMissing):
        _lib.load()


def test_ttt_attention_argument_checks_return_before_any_device_work(lib_path):
    """eagle_ttt_attn validates on the host and returns before touching the device:
    bad rounds and sizes give their status codes, an empty batch is a no-op (NULL
    pointers allowed), and misaligned pointers are refused.  No GPU is needed."""
    L = ctypes.CDLL(lib_path)
    f = L.eagle_ttt_attn
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_void_p,
                                                                ctypes.c_void_p]
    OK, INVALID, SHAPE = 0, 1, 2
    p = 4096                                      # a 16-byte aligned, never dereferenced address
    # B, S, Hq, Hkv, head_dim, R1, r, scale
    assert f(None, None, None, None, 0, 8, 4, 2, 128, 3, 1, 0.1, None, None) == OK
    assert f(p, p, p, p, 1, 8, 4, 2, 128, 3, 3, 0.1, None, None) == INVALID     # r >= R1
    assert f(p, p, p, p, 1, 8, 4, 2, 128, 3, -1, 0.1, None, None) == INVALID    # r < 0
    assert f(p, p, p, p, 1, 0, 4, 2, 128, 3, 1, 0.1, None, None) == INVALID     # S < 1
    assert f(p, p, p, p, 1, 8, 4, 2, 128, 3, 1, 0.0, None, None) == INVALID     # scale
    assert f(p, p, p, p, 1, 8, 4, 2, 64, 3, 1, 0.1, None, None) == SHAPE        # head_dim
    assert f(p, p, p, p, 1, 8, 4, 3, 128, 3, 1, 0.1, None, None) == SHAPE       # Hq % Hkv
    assert f(p, p, p, p, 1, 8, 4, 2, 128, 17, 1, 0.1, None, None) == SHAPE      # R1 > 16
    assert f(None, p, p, p, 1, 8, 4, 2, 128, 3, 1, 0.1, None, None) == INVALID  # NULL q
    assert f(p + 4, p, p, p, 1, 8, 4, 2, 128, 3, 1, 0.1, None, None) == INVALID  # misaligned


def test_filtered_verify_rejects_bad_filter_parameters(lib_path):
    """top_k < 0 and a negative or non-finite top_p are refused on the host; with valid
    parameters an empty batch returns OK without device work (the positive control).
    Arguments are placed by the parameter names the header declares."""
    import re
    from eagle_tree_speculative_gb300 import _lib
    L = ctypes.CDLL(lib_path)
    f = L.eagle_verify_accept_filtered
    f.restype = ctypes.c_int
    f.argtypes = _lib.SIGNATURES["eagle_verify_accept_filtered"][1]
    text = open(HEADER).read()
    decl = re.search(r"eagle_status eagle_verify_accept_filtered\((.*?)\);", text, re.S).group(1)
    params = [x.strip().split()[-1].lstrip("*") for x in decl.replace("\n", " ").split(",")]
    assert len(params) == len(f.argtypes)
    p = 4096                                      # a 16-byte aligned, never dereferenced address

    def run(top_k, top_p):
        vals = {"B": 0, "n": 2, "V": 8, "R": 2, "max_depth": 1, "temperature": 1.0, "seed": 0,
                "top_k": top_k, "top_p": top_p, "ws_bytes": 0}
        return f(*[vals.get(nm, p) for nm in params])

    assert run(5, 0.5) == 0
    assert run(-1, 0.5) == 1
    assert run(5, -0.1) == 1
    assert run(5, float("inf")) == 1
    assert run(5, float("nan")) == 1


def test_static_state_entry_reports_the_same_argument_errors(lib_path):
    """eagle2_expand_static_state checks its arguments on the host, like eagle2_expand and
    before any device call, so the two entry points give the same status for the same bad
    argument (no GPU is needed for that)."""
    L = ctypes.CDLL(lib_path)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    ex = L.eagle2_expand
    ex.restype = I
    ex.argtypes = [I, I, P, P, P, I, I, I, I, I, I, P, SZ, P, SZ, P, P, P, P, P, P]
    st = L.eagle2_expand_static_state
    st.restype = I
    st.argtypes = [I, I, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P]
    p = 4096                                        # never dereferenced
    cases = [  # level, final, B, V, top_k, depth, n_out
        (1, 0, -1, 100, 10, 8, 60),                 # B < 0
        (1, 0, 4, 100, 0, 8, 60),                   # top_k = 0
        (1, 0, 4, 100, 17, 8, 60),                  # top_k above the limit
        (1, 0, 4, 100, 10, 0, 60),                  # depth = 0
        (1, 0, 4, 5, 10, 8, 60),                    # top_k > V
        (9, 0, 4, 100, 10, 8, 60),                  # level beyond depth
        (1, 1, 4, 100, 10, 8, 65),                  # n_out above 64
        (2, 1, 4, 100, 10, 8, 200),                 # n_out above the candidates
    ]
    for lvl, fin, B, V, k, D, n in cases:
        a = ex(lvl, fin, None, None, p, B, 0, V, k, D, n, p, 1 << 40, None, 0, p, p, p, None,
               None, None)
        b = st(lvl, fin, None, None, p, B, 0, V, k, D, n, p, p, p, None, None, None)
        assert a == b and a != 0, (lvl, fin, B, V, k, D, n, a, b)


def test_every_call_treats_an_empty_batch_as_a_no_op(lib_path):
    """B == 0 (rows == 0, M == 0, n_layers == 0) with valid sizes returns OK before any
    device work, with every device pointer NULL; the same sizes with B = 1 and NULL
    pointers are refused, so the no-op is the empty batch's, not a missing check."""
    from eagle_tree_speculative_gb300 import _lib
    L = ctypes.CDLL(lib_path)
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    OK, INVALID = 0, 1
    N = None
    begin = (ctypes.c_int * 3)(0, 300, 1000)
    shards = (ctypes.c_void_p * 2)(None, None)
    calls = {
        # q k v kv_len parent out | B n Hq Hkv d Lmax scale | ws ws_bytes status stream
        "eagle_tree_attn": lambda B: L.eagle_tree_attn(N, N, N, N, N, N, B, 60, 32, 8, 128, 4156,
                                                       0.088, N, 0, N, N),
        "eagle_ttt_attn": lambda B: L.eagle_ttt_attn(N, N, N, N, B, 64, 4, 2, 128, 3, 1, 0.1, N, N),
        # tgt drf row tok par | B n V R D T seed | acc path emit stats status stream
        "eagle_verify_accept": lambda B: L.eagle_verify_accept(N, N, N, N, N, B, 60, 1000, 60, 8,
                                                               1.0, 0, N, N, N, N, N, N),
        "eagle_verify_accept_d2t": lambda B: L.eagle_verify_accept_d2t(
            N, N, N, N, N, B, 60, 1000, 60, 500, N, 8, 1.0, 0, N, N, N, N, N, N),
        "eagle_verify_accept_filtered": lambda B: L.eagle_verify_accept_filtered(
            N, N, N, N, N, B, 60, 1000, 60, 8, 1.0, 0, 20, 0.9, N, N, N, N, N, 0, N, N),
        "eagle_verify_accept_sharded": lambda B: L.eagle_verify_accept_sharded(
            shards, shards, begin, 2, N, N, N, B, 60, 1000, 60, 8, 1.0, 0, N, N, N, N, N, N),
        # k v kv_len path acc | n_layers B Hkv d Lmax D | status stream
        "eagle_kv_compact": lambda B: L.eagle_kv_compact(N, N, N, N, N, 32, B, 8, 128, 4160, 8,
                                                         N, N),
        # level final hidden w logits B H V k D n_out state bytes partials bytes out... status stream
        "eagle2_expand": lambda B: L.eagle2_expand(3, 1, N, N, N, B, 0, 1000, 10, 3, 60, N, 0, N, 0,
                                                   N, N, N, N, N, N),
        "eagle2_expand_d2t": lambda B: L.eagle2_expand_d2t(3, 1, N, N, N, B, 0, 1000, 10, 3, 60, N,
                                                           0, N, 0, N, N, N, N, N, N, N),
        "eagle2_expand_static_state": lambda B: L.eagle2_expand_static_state(
            3, 1, N, N, N, B, 0, 1000, 10, 3, 60, N, N, N, N, N, N),
        "eagle2_tree_candidates": lambda B: L.eagle2_tree_candidates(N, 0, B, 10, 3, N, N, N, N, N,
                                                                     N, N),
        "eagle_static_tree_level": lambda B: L.eagle_static_tree_level(2, N, N, N, N, N, 26, B, 26,
                                                                       1000, N, N, N),
        "eagle_softmax_stats": lambda B: L.eagle_softmax_stats(N, B, 1000, 1.0, N, N, N, N, N),
        "eagle_lmhead_gemm": lambda B: L.eagle_lmhead_gemm(N, N, N, B, 4096, 1000, 1000, 1, 0, 0,
                                                           N, N, N),
    }
    for name, call in calls.items():
        assert call(0) == OK, name
        assert call(1) == INVALID, name
