"""ctypes loader for libeagle_gb300.so: one declaration per entry point of include/eagle.h.

There is no fallback: if the compiled library is absent, loading raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libeagle_gb300.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/eagle.h
SIGNATURES = {
    "eagle_tree_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "eagle_tree_attn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P]),
    "eagle_ttt_attn": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P]),
    "eagle_verify_accept": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _U64, _P, _P, _P, _P,
                                 _P, _P]),
    "eagle_verify_filter_workspace_size": (_SZ, [_I, _I, _I]),
    "eagle_verify_accept_filtered": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _U64, _I,
                                          _F, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "eagle_verify_accept_sharded": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _F, _U64,
                                         _P, _P, _P, _P, _P, _P]),
    "eagle_d2t_inverse": (_I, [_P, _I, _I, _P, _P, _P]),
    "eagle_verify_accept_d2t": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _F, _U64, _P,
                                     _P, _P, _P, _P, _P]),
    "eagle_kv_compact": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "eagle2_tree_state_size": (_SZ, [_I, _I, _I]),
    "eagle2_expand_scratch_size": (_SZ, [_I, _I, _I]),
    "eagle2_expand": (_I, [_I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _SZ, _P, _P, _P,
                           _P, _P, _P]),
    "eagle2_expand_d2t": (_I, [_I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _SZ, _P, _P,
                               _P, _P, _P, _P, _P]),
    "eagle2_tree_candidates": (_I, [_P, _SZ, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "eagle_static_tree": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "eagle_static_tree_level": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "eagle2_expand_static_state": (_I, [_I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                        _P, _P]),
    "eagle_softmax_stats": (_I, [_P, _I64, _I, _F, _P, _P, _P, _P, _P]),
    "eagle_lmhead_gemm": (_I, [_P, _P, _P, _I, _I, _I, _I64, _I, _I64, _I64, _P, _P, _P]),
    "eagle_wait_selftest": (_I, [_P, _I64, _P]),
    "eagle_status_str": (ctypes.c_char_p, [_I]),
    "eagle_abi_version": (_I, []),
}

_lib = None


class LibraryMissing(RuntimeError):
    pass


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LibraryMissing(
                f"{LIB_PATH} not found: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib
