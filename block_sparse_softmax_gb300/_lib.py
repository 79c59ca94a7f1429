"""ctypes loader for libbss_attn.so: one Python function per C entry point,
same names, plain integers/pointers in, a status code out.

Nothing here computes: arguments are marshalled (device pointers, sizes, the
current CUDA stream) and the library does all the work.  Loading fails loudly
when the shared library has not been built.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

_C = ctypes
_SIGNATURES = {
    "attn_status_string": (_C.c_char_p, [_C.c_int]),
    "attn_last_error_message": (_C.c_char_p, []),
    "attn_version": (_C.c_int, []),
    "attn_fwd": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                            _C.c_int, _C.c_int, _C.c_int, _C.c_int, _C.c_int, _C.c_int,
                            _C.c_float, _C.c_int, _C.c_int64, _C.c_int64, _C.c_void_p]),
    "attn_fwd_partial": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                    _C.c_void_p, _C.c_void_p, _C.c_int, _C.c_int, _C.c_int,
                                    _C.c_int, _C.c_int, _C.c_int, _C.c_float, _C.c_int,
                                    _C.c_int64, _C.c_int64, _C.c_void_p]),
    "attn_merge_states": (_C.c_int, [_C.c_int, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                     _C.c_void_p, _C.c_void_p, _C.c_int, _C.c_int, _C.c_int,
                                     _C.c_int, _C.c_void_p]),
    "attn_fwd_splitkv_workspace_bytes": (_C.c_size_t, [_C.c_int, _C.c_int, _C.c_int, _C.c_int,
                                                       _C.c_int, _C.c_int]),
    "attn_fwd_splitkv": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                    _C.c_void_p, _C.c_void_p, _C.c_size_t, _C.c_int, _C.c_int,
                                    _C.c_int, _C.c_int, _C.c_int, _C.c_int, _C.c_float, _C.c_int,
                                    _C.c_int64, _C.c_int64, _C.c_int, _C.c_void_p]),
    "attn_select_blocks_workspace_bytes": (_C.c_size_t, [_C.c_int, _C.c_int, _C.c_int, _C.c_int]),
    "attn_select_blocks_nnz": (_C.c_int64, [_C.c_int, _C.c_int, _C.c_int, _C.c_int, _C.c_int]),
    "attn_select_blocks": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_int, _C.c_int, _C.c_int,
                                      _C.c_int, _C.c_int, _C.c_float, _C.c_int, _C.c_int,
                                      _C.c_int, _C.c_int, _C.c_int, _C.c_void_p, _C.c_void_p,
                                      _C.c_void_p, _C.c_size_t, _C.c_void_p]),
    "attn_blocklist_normalize": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_int, _C.c_int,
                                            _C.c_void_p, _C.c_void_p, _C.c_void_p]),
    "attn_blocklist_stats": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_int, _C.c_int, _C.c_int,
                                        _C.c_int, _C.c_int, _C.c_int, _C.c_void_p, _C.c_void_p]),
    "attn_fwd_blocksparse": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                        _C.c_void_p, _C.c_int, _C.c_int, _C.c_int, _C.c_int,
                                        _C.c_int, _C.c_float, _C.c_int, _C.c_int, _C.c_void_p,
                                        _C.c_void_p, _C.c_int, _C.c_int, _C.c_int, _C.c_void_p]),
    "attn_bwd_workspace_bytes": (_C.c_size_t, [_C.c_int, _C.c_int, _C.c_int, _C.c_int]),
    "attn_bwd": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                            _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                            _C.c_void_p, _C.c_size_t, _C.c_int, _C.c_int, _C.c_int, _C.c_int,
                            _C.c_int, _C.c_float, _C.c_int, _C.c_void_p]),
    "attn_bwd_blocksparse_workspace_bytes": (_C.c_size_t, [_C.c_int, _C.c_int, _C.c_int,
                                                           _C.c_int, _C.c_int]),
    "attn_bwd_blocksparse": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                        _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                        _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_size_t,
                                        _C.c_int, _C.c_int, _C.c_int, _C.c_int, _C.c_int,
                                        _C.c_float, _C.c_int, _C.c_int, _C.c_void_p, _C.c_void_p,
                                        _C.c_int, _C.c_int, _C.c_int, _C.c_void_p]),
    "attn_bwd_noalloc": (_C.c_int, [_C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                    _C.c_void_p, _C.c_void_p, _C.c_void_p, _C.c_void_p,
                                    _C.c_void_p, _C.c_void_p, _C.c_int, _C.c_int, _C.c_int,
                                    _C.c_int, _C.c_int, _C.c_float, _C.c_int, _C.c_void_p]),
    "attn_poll_status": (_C.c_int, [_C.c_void_p]),
    "attn_bwd_time_main": (_C.c_int, [_C.c_void_p, _C.c_void_p]),
    "attn_watchdog_selftest": (_C.c_int, [_C.c_ulonglong, _C.c_void_p]),
    "attn_probe_ex2_rate": (_C.c_int, [_C.c_void_p, _C.c_int, _C.c_int, _C.c_void_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()' or python -m block_sparse_softmax_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (restype, argtypes) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = restype
            fn.argtypes = argtypes
        _lib = lib
    return _lib


def exported_names():
    return list(_SIGNATURES)
