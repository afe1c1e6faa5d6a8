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
    # header, 5 words per candidate (711 at k=10, D=8), frontier, and per (row, segment)
    # of up to 4 vocabulary segments: 3 statistics words + k values + k tokens
    assert E.tree_state_size(64, 10, 8) == 64 * 4 * (4 + 5 * 711 + 16 + 10 * 4 * (3 + 2 * 10))
    assert E.tree_state_size(1, 17, 8) == 0                # top_k above the limit
    assert E.tree_attn_workspace_size(64, 60, 32, 8, 128, 4156) >= 0
    assert E.tree_attn_workspace_size(1, 60, 32, 8, 64, 4156) == 0    # head_dim != 128


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from eagle_tree_speculative_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(_lib.LibraryMissing):
        _lib.load()
