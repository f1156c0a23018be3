"""ctypes view of libsa.so (include/sa.h).  Loading fails loudly when the
library has not been built: there is no other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsa.so")

SA_OK = 0
STATUS_NAMES = {
    0: "OK", 1: "HEAD_COUNT", 2: "BLOCK_PAGE", 3: "CU_SEQLENS", 4: "SHAPE",
    5: "SELECTED_RANGE", 6: "HEAD_DIM", 7: "EMPTY", 8: "CUDA", 9: "DEVICE_TIMEOUT",
    10: "UNSUPPORTED", 11: "INVALID_ARGUMENT",
}
DTYPE_F32, DTYPE_BF16 = 0, 1
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR_CORE, PATH_CUDA_CORE_GENERAL, PATH_FUSED_DECODE = 0, 1, 2, 3, 4
PATH_TENSOR_CORE_TF32 = 5

#: Every symbol include/sa.h declares.
EXPORTS = ("sa_status_string", "sa_version", "sa_index_query_sizes", "sa_index_workspace_size",
           "sa_build_index",
           "sa_build_index_no_alloc", "sa_forward", "sa_forward_ex", "sa_forward_combine",
           "sa_forward_combine_ex", "sa_forward_kernel_name", "sa_attention_kernel_name",
           "sa_combine", "sa_combine_ex", "sa_attention", "sa_attention_ex", "sa_get_status",
           "sa_clear_status", "sa_debug_stall", "sa_debug_cta_stats")


class SaIndex(ctypes.Structure):
    _fields_ = [
        ("tq", ctypes.c_int64),
        ("hkv", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("pages_per_block", ctypes.c_int32),
        ("msb", ctypes.c_int32),
        ("nbs", ctypes.c_int64),
        ("split_edges", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("sel_slots", ctypes.c_void_p),
        ("sel_offsets", ctypes.c_void_p),
        ("num_sel", ctypes.c_void_p),
        ("edge_head_base", ctypes.c_void_p),
        ("edges", ctypes.c_void_p),
        ("inv", ctypes.c_void_p),
        ("splits", ctypes.c_void_p),
        ("totals", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class SaIndexSizes(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in
                ("msb", "nbs", "sel_slots", "sel_offsets", "num_sel", "edge_head_base",
                 "edges", "inv", "splits", "totals")] + [("workspace_bytes", ctypes.c_size_t)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -m block_sparse_paged_csr_gb300.build "
            "or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    p, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    st = ctypes.c_int
    lib.sa_status_string.argtypes = [st]
    lib.sa_status_string.restype = ctypes.c_char_p
    lib.sa_version.argtypes = []
    lib.sa_version.restype = ctypes.c_char_p
    lib.sa_index_query_sizes.argtypes = [i64, i32, i32, i32, i32, i32, i32,
                                         ctypes.POINTER(SaIndexSizes)]
    lib.sa_index_query_sizes.restype = st
    lib.sa_index_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32, i32,
                                            ctypes.POINTER(ctypes.c_size_t)]
    lib.sa_index_workspace_size.restype = st
    lib.sa_build_index.argtypes = [p, i64, i32, i32, p, p, i32, p, i32, i32, i32, i32,
                                   ctypes.POINTER(SaIndex), p]
    lib.sa_build_index.restype = st
    lib.sa_build_index_no_alloc.argtypes = lib.sa_build_index.argtypes
    lib.sa_build_index_no_alloc.restype = st
    lib.sa_forward.argtypes = [p, p, p, i64, st, ctypes.POINTER(SaIndex), p, p, p, i32, i32, i32,
                               i32, i32, f32, i32, p, p, p, st, p]
    lib.sa_forward.restype = st
    lib.sa_forward_ex.argtypes = [p, p, p, i64, st, ctypes.POINTER(SaIndex), p, p, p, i32, i32,
                                  i32, i32, i32, f32, i32, st, p, p, p, st, p, p]
    lib.sa_forward_ex.restype = st
    lib.sa_forward_combine.argtypes = [p, p, p, i64, st, ctypes.POINTER(SaIndex), p, p, p, p, p,
                                       i32, i32, i32, i32, f32, i32, i32, p, p, p, p, p, st, p]
    lib.sa_forward_combine.restype = st
    lib.sa_forward_combine_ex.argtypes = [p, p, p, i64, st, ctypes.POINTER(SaIndex), p, p, p, p,
                                          p, i32, i32, i32, i32, f32, i32, i32, st, p, p, p, p,
                                          p, st, p]
    lib.sa_forward_combine_ex.restype = st
    lib.sa_forward_kernel_name.argtypes = [i64, i32, i32, i32, i32, i32, i32, st, st]
    lib.sa_forward_kernel_name.restype = ctypes.c_char_p
    lib.sa_attention_kernel_name.argtypes = [i64, i32, p, i64, i32, i32, i32, i32, i32, st, i32,
                                             st]
    lib.sa_attention_kernel_name.restype = ctypes.c_char_p
    lib.sa_combine.argtypes = [ctypes.POINTER(SaIndex), p, p, p, i32, i32, p, p, p]
    lib.sa_combine.restype = st
    lib.sa_combine_ex.argtypes = [ctypes.POINTER(SaIndex), st, p, p, p, i32, i32, p, p, p]
    lib.sa_combine_ex.restype = st
    lib.sa_attention.argtypes = [p, p, p, i64, st, p, i64, i32, p, p, i32, p, p, i32, i32, i32,
                                 i32, i32, i32, f32, i32, i32, ctypes.POINTER(SaIndex), p, p, p,
                                 p, p, st, p]
    lib.sa_attention.restype = st
    lib.sa_attention_ex.argtypes = [p, p, p, i64, st, p, i64, i32, p, p, i32, p, p, i32, i32,
                                    i32, i32, i32, i32, f32, i32, i32, ctypes.POINTER(SaIndex),
                                    st, p, p, p, p, p, st, p]
    lib.sa_attention_ex.restype = st
    lib.sa_get_status.argtypes = [ctypes.POINTER(SaIndex), p]
    lib.sa_get_status.restype = st
    lib.sa_clear_status.argtypes = [ctypes.POINTER(SaIndex), p]
    lib.sa_clear_status.restype = st
    lib.sa_debug_stall.argtypes = [i32, ctypes.c_uint32]
    lib.sa_debug_stall.restype = st
    lib.sa_debug_cta_stats.argtypes = [p, i32]
    lib.sa_debug_cta_stats.restype = st
    if path == LIB_PATH:
        _lib = lib
    return lib
