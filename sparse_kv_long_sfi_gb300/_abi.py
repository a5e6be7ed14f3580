"""ctypes view of include/sfi.h: the structures and prototypes of libsfi.

Loading fails loudly when the library has not been built: there is no other
implementation of these calls in this package.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_u32 = ctypes.c_uint32


class sfi_attn_shape(ctypes.Structure):
    _fields_ = [("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32), ("page_size", c_i32),
                ("softmax_scale", c_f32)]


class sfi_paged_kv(ctypes.Structure):
    _fields_ = [("k_pool", c_vp), ("v_pool", c_vp), ("num_pages", c_i32), ("max_pages_per_req", c_i32),
                ("page_table", c_vp), ("seq_lens", c_vp)]


class sfi_compact_kv(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("total_rows", c_i64), ("row_offset", c_vp), ("capacity", c_vp),
                ("count", c_vp)]


SFI_OK, SFI_ERR_INVALID_ARG, SFI_ERR_UNSUPPORTED, SFI_ERR_WORKSPACE, SFI_ERR_CUDA = range(5)
SFI_DEV_BAD_PAGE, SFI_DEV_BAD_LEN, SFI_DEV_K_OVERFLOW = 1, 2, 4
SFI_DEV_BAD_INDEX, SFI_DEV_TIMEOUT, SFI_DEV_BAD_COMPACT = 8, 16, 32
SFI_ATTN_EARLY_KV_PREFETCH = 1
SFI_ATTN_RAGGED = 2
SFI_ATTN_TEST_WITHHOLD = 4
SFI_MAX_QUERY_TOKENS = 16

P_SHAPE = ctypes.POINTER(sfi_attn_shape)
P_PAGED = ctypes.POINTER(sfi_paged_kv)
P_COMPACT = ctypes.POINTER(sfi_compact_kv)

# name -> (restype, argtypes), in the order of include/sfi.h
PROTOTYPES = {
    "sfi_paged_kv_append": (c_i32, [P_SHAPE, P_PAGED, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp]),
    "sfi_fast_decode_attn": (c_i32, [P_SHAPE, P_PAGED, P_COMPACT, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                     c_vp, c_i32, c_i32, c_i32, c_u32, c_vp, c_sz, c_vp, c_vp]),
    "sfi_slow_dense_attn_with_scores": (c_i32, [P_SHAPE, P_PAGED, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                                c_i64, c_vp, c_i32, c_i32, c_i32, c_u32, c_vp, c_sz, c_vp, c_vp]),
    "sfi_mixed_decode_attn": (c_i32, [P_SHAPE, P_PAGED, P_COMPACT, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                      c_vp, c_i64, c_vp, c_i32, c_vp, c_i32, c_i32, c_i32, c_u32, c_vp, c_sz,
                                      c_vp, c_vp]),
    "sfi_mixed_workspace_size": (c_sz, [P_SHAPE, c_i32, c_i32, c_i32, c_i32]),
    "sfi_paged_kv_append_tokens": (c_i32, [P_SHAPE, P_PAGED, c_vp, c_vp, c_i32, c_vp, c_i32, c_vp, c_vp]),
    "sfi_dense_verify_attn": (c_i32, [P_SHAPE, P_PAGED, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                      c_i64, c_vp, c_i32, c_i32, c_i32, c_u32, c_vp, c_sz, c_vp, c_vp]),
    "sfi_sparse_draft_attn": (c_i32, [P_SHAPE, P_PAGED, P_COMPACT, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp,
                                      c_vp, c_i32, c_i32, c_i32, c_u32, c_vp, c_sz, c_vp, c_vp]),
    "sfi_multi_workspace_size": (c_sz, [P_SHAPE, c_i32, c_i32, c_i32, c_i32]),
    "sfi_select_topk": (c_i32, [c_vp, c_i64, c_i32, c_vp, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp, c_i32, c_vp,
                                c_vp]),
    "sfi_compact_gather": (c_i32, [P_SHAPE, P_PAGED, c_vp, c_vp, c_i32, c_i32, P_COMPACT, c_vp, c_i32, c_vp,
                                   c_vp]),
    "sfi_select_compact": (c_i32, [P_SHAPE, P_PAGED, c_vp, c_i64, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, P_COMPACT,
                                   c_vp, c_i32, c_vp, c_vp]),
    "sfi_fast_decode_attn_noalloc": (c_i32, [P_SHAPE, P_PAGED, P_COMPACT, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp,
                                             c_vp, c_vp, c_i32, c_i32, c_i32, c_u32, c_vp, c_vp]),
    "sfi_workspace_size": (c_sz, [P_SHAPE, c_i32, c_i32, c_i32]),
    "sfi_plan_splits": (c_i32, [P_SHAPE, c_i32, c_i32, c_i32]),
    "sfi_attn_cluster_capacity": (c_i32, [c_i32]),
    "sfi_status_string": (ctypes.c_char_p, [c_i32]),
    "sfi_version": (c_i32, []),
}

_lock = threading.Lock()
_lib = None


def lib(path: str = LIB):
    """The loaded libsfi (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libsfi.so is not built ({path}); run sparse_kv_long_sfi_gb300.build.build() first")
            L = ctypes.CDLL(path)
            for name, (res, args) in PROTOTYPES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib
