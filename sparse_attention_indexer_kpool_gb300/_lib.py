"""ctypes loader for libdsa.so (the C ABI declared in include/dsa.h).

The library is built in-tree by ``build.py``; if it is missing the first call
raises: there is no CPU fallback anywhere in the product path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LIB = None
_LOCK = threading.Lock()

c_void_p, c_int, c_float, c_size_t = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class DecodeLayerArgs(ctypes.Structure):
    """dsa_decode_layer_args (include/dsa.h), field for field."""
    _fields_ = [(n, c_void_p) for n in ("k", "gate", "valid", "ape", "ln_gamma", "ln_beta")] + [
        ("ln_eps", c_float), ("cu_seqlens", c_void_p), ("pool_begin", c_void_p),
        ("max_pools", c_int), ("pool_keys", c_void_p), ("pool_rows", c_int),
        ("pool_start", c_void_p), ("pool_valid", c_void_p), ("n_pools", c_void_p),
        ("cu_pool_cap", c_void_p), ("q", c_void_p), ("weights", c_void_p), ("scale", c_float),
        ("q_seq", c_void_p), ("q_pos", c_void_p), ("q_lat", c_void_p), ("kv_latent", c_void_p),
        ("sm_scale", c_float)] + [(n, c_int) for n in (
            "Q", "B", "H", "D", "kpool", "P_ld", "select_k", "out_width", "Hm", "L", "dtype")] + [
        (n, c_void_p) for n in ("scores", "pool_ids", "token_ids", "out", "lse", "ws_select")] + [
        ("ws_select_bytes", c_size_t), ("ws_mla", c_void_p), ("ws_mla_bytes", c_size_t),
        ("status_dev", c_void_p)]


class PagedKv(ctypes.Structure):
    """dsa_paged_kv (include/dsa.h), field for field."""
    _fields_ = [(n, c_void_p) for n in ("pages", "row_scale", "block_table", "seq_lens")] + [
        (n, c_int) for n in ("n_pages", "page_size", "max_pages", "kv_dtype")]


# name -> (restype, argtypes); mirrors include/dsa.h
SIGNATURES = {
    "dsa_kpool_compress": (c_int, [c_void_p] * 6 + [c_float] + [c_void_p] * 3 + [c_int] * 5
                           + [c_void_p] * 6),
    "dsa_index_scores": (c_int, [c_void_p, c_void_p, c_float, c_void_p, c_int] + [c_void_p] * 6
                         + [c_int] * 7 + [c_void_p] * 3),
    "dsa_topk_pools": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_size_t,
                               c_void_p]),
    "dsa_topk_pools_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "dsa_expand_selection": (c_int, [c_void_p] * 4 + [c_int] * 5 + [c_void_p] * 3),
    "dsa_mla_selected_decode": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int]
                                + [c_void_p] * 3 + [c_size_t] + [c_void_p] * 2),
    "dsa_mla_selected_decode_workspace_size": (c_size_t, [c_int] * 5),
    "dsa_mla_paged_decode": (c_int, [c_void_p, ctypes.POINTER(PagedKv), c_void_p, c_void_p]
                             + [c_int] * 5 + [c_float, c_int] + [c_void_p] * 3 + [c_size_t]
                             + [c_void_p] * 2),
    "dsa_mla_paged_decode_workspace_size": (c_size_t, [c_int] * 6),
    "dsa_select": (c_int, [c_void_p, c_void_p, c_float, c_void_p, c_int] + [c_void_p] * 6
                   + [c_int] * 9 + [c_void_p] * 4 + [c_size_t] + [c_void_p] * 2),
    "dsa_select_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "dsa_select_noalloc": (c_int, [c_void_p, c_void_p, c_float, c_void_p, c_int]
                           + [c_void_p] * 6 + [c_int] * 9 + [c_void_p] * 5),
    "dsa_decode_layer": (c_int, [ctypes.POINTER(DecodeLayerArgs), c_void_p]),
    "dsa_decode_layer_workspace_size": (c_size_t, [ctypes.POINTER(DecodeLayerArgs),
                                                   ctypes.POINTER(c_size_t),
                                                   ctypes.POINTER(c_size_t)]),
    "dsa_status_string": (ctypes.c_char_p, [c_int]),
    "dsa_version": (c_int, []),
    "dsa_kernel_launches": (ctypes.c_uint64, []),
    "dsa_set_failure_drill": (c_int, [c_int]),
    "dsa_indexer_project": (c_int, [c_void_p] * 5 + [c_int] * 8 + [c_float] + [c_void_p] * 8
                            + [c_size_t] + [c_void_p] * 2),
    "dsa_indexer_project_workspace_size": (c_size_t, [c_int] * 8),
}


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libdsa.so once; raise if it is not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = lib_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"libdsa.so is not built ({path}); run "
                    "`python -m sparse_attention_indexer_kpool_gb300.build` (needs nvcc)")
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB
