"""ctypes binding of libattnbwd.so.  Same names and arguments as include/attnbwd.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these symbols.  Loading fails loudly when the library has not
been built (``python -m attention_backward_02_gb300.build`` or
``__graft_entry__.build()``); there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libattnbwd.so")

ATTN_OK, ATTN_ERR_NULLPTR, ATTN_ERR_INVALID, ATTN_ERR_UNSUPPORTED = 0, 1, 2, 3
ATTN_ERR_WORKSPACE, ATTN_ERR_ALIGN, ATTN_ERR_CUDA, ATTN_ERR_DEVICE = 4, 5, 6, 7
ATTN_DEV_TIMEOUT, ATTN_DEV_INDEX_RANGE, ATTN_DEV_INDEX_DUP = 0x1, 0x2, 0x4
ATTN_F16, ATTN_BF16 = 0, 1
ATTN_MASK_NONE, ATTN_CAUSAL_TOP_LEFT, ATTN_CAUSAL_BOTTOM_RIGHT = 0, 1, 2
ATTN_DQ_ATOMIC, ATTN_DQ_SPLIT, ATTN_DQ_ORDERED = 0, 1, 2

# every exported symbol of include/attnbwd.h
EXPORTS = ("sdpa_workspace_size", "sdpa_fwd_stats", "sdpa_bwd", "nsa_workspace_size",
           "nsa_selected_attn_bwd", "nsa_block_lists", "attn_query_status", "attn_status_string",
           "attn_set_main_kernel_events", "sdpa_bwd_static_scratch", "attn_static_scratch_status",
           "attn_selftest_wait_timeout", "attn_selftest_occupy", "attn_last_error",
           "nsa_fwd_workspace_size", "nsa_selected_attn_fwd")


class attn_view_t(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("sb", C.c_int64), ("sh", C.c_int64), ("ss", C.c_int64)]


class attn_sdpa_desc_t(C.Structure):
    _fields_ = [("dtype", C.c_int), ("b", C.c_int64), ("h", C.c_int64), ("h_kv", C.c_int64),
                ("s_q", C.c_int64), ("s_kv", C.c_int64), ("d", C.c_int64), ("scale", C.c_double),
                ("mask", C.c_int), ("cu_seqlens_q", C.POINTER(C.c_int64)),
                ("cu_seqlens_kv", C.POINTER(C.c_int64)), ("deterministic", C.c_int), ("dq_splits", C.c_int)]


class attn_nsa_desc_t(C.Structure):
    _fields_ = [("dtype", C.c_int), ("b", C.c_int64), ("cu_seqlens_q", C.POINTER(C.c_int64)),
                ("cu_seqlens_kv", C.POINTER(C.c_int64)), ("n1", C.c_int64), ("n2", C.c_int64),
                ("d", C.c_int64), ("scale", C.c_double), ("block_size", C.c_int64),
                ("block_count", C.c_int64), ("sparse_mode", C.c_int), ("deterministic", C.c_int),
                ("d_v", C.c_int64), ("grad_fp32", C.c_int), ("atten_mask", C.c_void_p),
                ("mask_rows", C.c_int64), ("mask_cols", C.c_int64)]


_lib = None


def load() -> C.CDLL:
    """Load the built library and declare the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libattnbwd.so is not built ({LIB_PATH} missing); run __graft_entry__.build() "
                          "or python -m attention_backward_02_gb300.build")
    lib = C.CDLL(LIB_PATH)
    P, V, S, I = C.POINTER, C.c_void_p, C.c_size_t, C.c_int
    D, N, view = P(attn_sdpa_desc_t), P(attn_nsa_desc_t), attn_view_t
    sig = {
        "sdpa_workspace_size": [D, P(S), P(S)],
        "sdpa_fwd_stats": [D, view, view, view, view, P(C.c_float), V, S, V],
        "sdpa_bwd": [D, view, view, view, view, view, P(C.c_float), view, view, view, V, S, V],
        "nsa_workspace_size": [N, P(S)],
        "nsa_fwd_workspace_size": [N, P(S)],
        "nsa_selected_attn_fwd": [N, V, V, V, P(C.c_int32), V, P(C.c_float), P(C.c_float), V, S, V],
        "nsa_selected_attn_bwd": [N, V, V, V, V, V, P(C.c_float), P(C.c_float), P(C.c_int32), V, V, V, V, S, V],
        "nsa_block_lists": [N, P(C.c_int32), P(C.c_int32), P(C.c_int32), P(C.c_int64), V, S, V],
        "attn_query_status": [V, V, P(C.c_uint32)],
        "attn_status_string": [I],
        "attn_last_error": [],
        "attn_set_main_kernel_events": [V, V],
        "sdpa_bwd_static_scratch": [D, view, view, view, view, view, P(C.c_float), view, view, view, V],
        "attn_static_scratch_status": [V, P(C.c_uint32)],
        "attn_selftest_wait_timeout": [V, S, C.c_double, V],
        "attn_selftest_occupy": [I, S, C.c_double, V],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_char_p if name in ("attn_status_string", "attn_last_error") else I
    _lib = lib
    return lib


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = load().attn_status_string(status).decode()
        detail = load().attn_last_error().decode() if status == ATTN_ERR_CUDA else ""
        super().__init__(f"{where} returned {name} ({status})" + (f": {detail}" if detail else ""))


def check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)
