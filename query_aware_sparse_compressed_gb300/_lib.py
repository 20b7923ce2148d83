"""ctypes view of libqasc's C ABI (include/qasc.h).  Marshalling only."""

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqasc.so")

QASC_OK = 0
QASC_ERR_INVALID_ARG = 1
STATUS_NAMES = {0: "QASC_OK", 1: "QASC_ERR_INVALID_ARG", 2: "QASC_ERR_UNSUPPORTED", 3: "QASC_ERR_WORKSPACE",
                4: "QASC_ERR_CUDA", 5: "QASC_ERR_TIMEOUT", 6: "QASC_ERR_BAD_TABLE",
                7: "QASC_ERR_INTERNAL"}


class qasc_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("d_idx", ctypes.c_int32), ("reserved", ctypes.c_int32), ("n", ctypes.c_int64),
                ("n_cap", ctypes.c_int64)]


class qasc_ts_params(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int32), ("sink", ctypes.c_int32), ("local", ctypes.c_int32), ("vmin", ctypes.c_int32)]


class qasc_snap_params(ctypes.Structure):
    _fields_ = [("c", ctypes.c_int32), ("window", ctypes.c_int32), ("pool_k", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class qasc_paged_cache(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("page_tokens", ctypes.c_int32), ("pages_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int64)]


class qasc_local_ring(ctypes.Structure):
    _fields_ = [("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("ring_tokens", ctypes.c_int32)]


_P = ctypes.c_void_p
_SP = ctypes.POINTER(qasc_shape)
_TP = ctypes.POINTER(qasc_ts_params)
_NP = ctypes.POINTER(qasc_snap_params)
_PC = ctypes.POINTER(qasc_paged_cache)
_RG = ctypes.POINTER(qasc_local_ring)

# name -> (restype, argtypes)
SIGNATURES = {
    "ts_index_append": (ctypes.c_int, [_SP, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, _P]),
    "ts_select_workspace_bytes": (ctypes.c_size_t, [_SP, _TP]),
    "ts_score_vote_select": (ctypes.c_int, [_SP, _TP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ts_attn_workspace_bytes": (ctypes.c_size_t, [_SP, _TP]),
    "ts_sparse_attn": (ctypes.c_int, [_SP, _TP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ts_sparse_attn_noalloc": (ctypes.c_int, [_SP, _TP, _P, _P, _P, _P, _P, _P, _P]),
    "ts_head_select_workspace_bytes": (ctypes.c_size_t, [_SP, _TP]),
    "ts_score_select_per_head": (ctypes.c_int, [_SP, _TP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ts_sparse_attn_per_head": (ctypes.c_int, [_SP, _TP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ts_expand_capacity": (ctypes.c_int32, [_SP, _TP, ctypes.c_int32]),
    "ts_expand_workspace_bytes": (ctypes.c_size_t, [_SP, _TP, ctypes.c_int32]),
    "ts_expand_neighbors": (ctypes.c_int, [_SP, _TP, ctypes.c_int32, _P, ctypes.c_int32, _P, ctypes.c_int32, _P,
                                           _P, ctypes.c_size_t, _P]),
    "ts_sparse_attn_ex": (ctypes.c_int, [_SP, _TP, _P, _P, _P, _P, _P, ctypes.c_int32, _P, _P, _P, ctypes.c_size_t,
                                         _P]),
    "ts_index_append_paged": (ctypes.c_int, [_SP, _PC, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, _P]),
    "ts_score_vote_select_paged": (ctypes.c_int, [_SP, _TP, _PC, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ts_score_select_per_head_paged": (ctypes.c_int, [_SP, _TP, _PC, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ts_sparse_attn_paged": (ctypes.c_int, [_SP, _TP, _PC, _RG, _P, _P, _P, _P, _P, ctypes.c_int32, _P, _P, _P,
                                            ctypes.c_size_t, _P]),
    "ts_ring_flush": (ctypes.c_int, [_SP, _PC, _RG, _P, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, _P]),
    "ts_dense_attn_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "ts_dense_attn": (ctypes.c_int, [_SP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "snapkv_workspace_bytes": (ctypes.c_size_t, [_SP, _NP]),
    "snapkv_compress": (ctypes.c_int, [_SP, _NP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qasc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qasc_last_error": (ctypes.c_char_p, []),
    "qasc_last_cuda_error": (ctypes.c_char_p, []),
    "qasc_device_error": (ctypes.c_int, [_P]),
    "qasc_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_int32, _P]),
    "qasc_version": (ctypes.c_int32, []),
}

_lib = None


def load(path=None):
    """Load libqasc.so (raises if it has not been built).  The environment
    variable QASC_LIB names another build to load instead, e.g. the
    NVTX-instrumented libqasc_nvtx.so."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or os.environ.get("QASC_LIB") or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libqasc.so is not built (%s); run query_aware_sparse_compressed_gb300.build.build()" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib
