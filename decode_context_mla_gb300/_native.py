"""ctypes declarations for libdcpmla (include/dcpmla.h).  Loads the in-tree library.

There is no CPU fallback: if the library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdcpmla.so")

i32, i64, f32, sz, vp = C.c_int32, C.c_int64, C.c_float, C.c_size_t, C.c_void_p
P_i32, P_i64 = C.POINTER(C.c_int32), C.POINTER(C.c_int64)
P_sz = C.POINTER(C.c_size_t)

# name -> (restype, argtypes); mirrors include/dcpmla.h
SIGNATURES = {
    "dcpmla_status_string": (C.c_char_p, [C.c_int]),
    "dcpmla_version": (C.c_int, []),
    "dcpmla_alloc_create": (C.c_int, [i32, i64, i32, vp, C.POINTER(vp)]),
    "dcpmla_alloc_destroy": (C.c_int, [vp]),
    "dcpmla_alloc_geometry": (C.c_int, [vp, P_i32, P_i32, P_i32, P_i64, P_i64]),
    "dcpmla_alloc_free_count": (C.c_int, [vp, P_i64]),
    "dcpmla_alloc_pages": (C.c_int, [vp, i32, vp]),
    "dcpmla_free_pages": (C.c_int, [vp, i32, vp]),
    "dcpmla_effective_page_size": (C.c_int, [vp, P_i32]),
    "dcpmla_reqmap_create": (C.c_int, [vp, i32, i32, C.POINTER(vp)]),
    "dcpmla_reqmap_destroy": (C.c_int, [vp]),
    "dcpmla_reqmap_extend": (C.c_int, [vp, i32, i64, P_i64]),
    "dcpmla_reqmap_release": (C.c_int, [vp, i32]),
    "dcpmla_reqmap_length": (C.c_int, [vp, i32, P_i64]),
    "dcpmla_reqmap_page_table": (C.c_int, [vp, vp, i32, i32, i32, vp, vp]),
    "dcpmla_map_positions": (C.c_int, [vp, i32, i32, i32, i32, vp, vp, i64, vp, vp, vp]),
    "dcpmla_slot_map": (C.c_int, [vp, i32, i32, i64, i32, i32, i32, vp, vp, i64, vp, vp, vp, vp,
                                  vp]),
    "dcpmla_kv_append": (C.c_int, [vp, vp, i32, i64, i32, vp, vp, vp, i64, vp, i64, vp, i64, vp,
                                   vp]),
    "dcpmla_decode": (C.c_int, [vp, vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                i32, i32, f32, i32, vp, vp, vp, sz, vp, vp]),
    "dcpmla_decode_noalloc": (C.c_int, [vp, vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, i32,
                                        i32, i32, i32, f32, i32, vp, vp, vp, vp]),
    "dcpmla_decode_workspace_size": (C.c_int, [i32, i32, i32, i32, i32, i32, i32, i32, P_sz]),
    "dcpmla_decode_path": (C.c_int, [i32, i32, i32, i32, i32, i32, i32, i32, P_i32, P_i32]),
    "dcpmla_decode_merged_workspace_size": (C.c_int, [i32, i32, i32, i32, i32, i32, i32, P_sz]),
    "dcpmla_decode_merged": (C.c_int, [vp, vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                       f32, i32, vp, vp, vp, sz, vp, vp]),
    "dcpmla_lse_merge": (C.c_int, [vp, vp, i32, i64, i32, vp, vp, vp, vp]),
    "dcpmla_testing_set_wait_limit": (C.c_int, [i64]),
    "dcpmla_relayout_dense_to_striped": (C.c_int, [vp, vp, i64, vp, i32, vp, vp, i32, i64, vp, i32,
                                                   vp, i32, i32, i32, i32, vp, vp]),
    "dcpmla_gather_unstriped": (C.c_int, [vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, i32, vp, vp,
                                          i64, vp, vp]),
    "dcpmla_kv_append_e4m3": (C.c_int, [vp, vp, i64, i32, vp, vp, vp, i64, vp, i64, i64, vp, vp]),
    "dcpmla_hicache_filter_workspace_size": (C.c_int, [i64, P_sz]),
    "dcpmla_hicache_filter": (C.c_int, [vp, i64, i32, i32, i32, vp, vp, vp, sz, vp, vp]),
}

_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libdcpmla is not built ({LIB_PATH} missing). Build it with "
                "`python -m decode_context_mla_gb300.build`; there is no CPU fallback.")
        handle = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib
