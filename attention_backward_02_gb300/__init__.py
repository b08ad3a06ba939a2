"""GB300 (sm_103a) SDPA backward (FlashAttention-2 form) and NSA selected-attention
backward behind a C ABI (include/attnbwd.h).

The functions here marshal torch CUDA tensors into the C ABI: pointers,
strides, the caller's stream and a caller-sized workspace.  PyTorch only
provides device memory and streams; all arithmetic runs in the library's
CUDA kernels.
"""
from __future__ import annotations

import ctypes as C

from . import _lib
from ._lib import (ATTN_BF16, ATTN_CAUSAL_BOTTOM_RIGHT, ATTN_CAUSAL_TOP_LEFT, ATTN_DQ_ATOMIC, ATTN_DQ_ORDERED,
                   ATTN_DQ_SPLIT, ATTN_F16, ATTN_MASK_NONE, AttnError, attn_nsa_desc_t, attn_sdpa_desc_t, attn_view_t, check)

__all__ = ["sdpa_desc", "nsa_desc", "view_bhsd", "view_tnd", "sdpa_workspace_size", "sdpa_fwd_stats",
           "sdpa_bwd", "nsa_workspace_size", "nsa_selected_attn_bwd", "nsa_block_lists",
           "nsa_fwd_workspace_size", "nsa_selected_attn_fwd",
           "attn_query_status", "AttnError", "ATTN_F16", "ATTN_BF16", "ATTN_MASK_NONE",
           "ATTN_CAUSAL_TOP_LEFT", "ATTN_CAUSAL_BOTTOM_RIGHT"]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"fp16 or bf16 expected, got {t.dtype}")


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class _Keep:
    """Holds ctypes arrays alive for the duration of a call."""

    def __init__(self):
        self.items = []


def _cu_array(keep, cu):
    if cu is None:
        return None
    arr = (C.c_int64 * len(cu))(*[int(x) for x in cu])
    keep.items.append(arr)
    return C.cast(arr, C.POINTER(C.c_int64))


def sdpa_desc(*, dtype, b, h, h_kv, s_q, s_kv, d, scale, mask=ATTN_MASK_NONE, cu_seqlens_q=None,
              cu_seqlens_kv=None, deterministic=False, dq_splits=0, _keep=None):
    """An attn_sdpa_desc_t.  Fixed-length mode: b sequences of s_q queries and s_kv keys.  Packed
    (varlen) mode: cu_seqlens_q / cu_seqlens_kv, b inclusive cumulative lengths each (s_q, s_kv then
    ignored).  scale multiplies q.k; mask is ATTN_MASK_NONE, ATTN_CAUSAL_TOP_LEFT or
    ATTN_CAUSAL_BOTTOM_RIGHT.  deterministic: False / ATTN_DQ_ATOMIC, True / ATTN_DQ_SPLIT (dq_splits
    partial buffers, 0: a default) or ATTN_DQ_ORDERED (one buffer, adds in a fixed order); the last two
    make dQ bitwise reproducible.  The host arrays live as long as the descriptor."""
    keep = _keep if _keep is not None else _Keep()
    mode = int(deterministic) if not isinstance(deterministic, bool) else int(deterministic)
    desc = attn_sdpa_desc_t(int(dtype), int(b), int(h), int(h_kv), int(s_q), int(s_kv), int(d), float(scale),
                            int(mask), _cu_array(keep, cu_seqlens_q), _cu_array(keep, cu_seqlens_kv),
                            mode, int(dq_splits))
    desc._keep = keep
    return desc


def nsa_desc(*, dtype, cu_seqlens_q, cu_seqlens_kv, n1, n2, d, scale, block_size, block_count, sparse_mode,
             deterministic=False, d_v=0, grad_fp32=False, atten_mask=None):
    """An attn_nsa_desc_t: TND layout, b = len(cu_seqlens_q) sequences with inclusive cumulative query /
    key lengths, n1 query and n2 kv heads, query / key head dim d and value head dim d_v (0: d),
    scaleValue, selectedBlockSize / Count, sparseMode 0 (selection only) or 2 (also causal,
    bottom-right per sequence); deterministic makes dq, dk, dv bitwise reproducible (tensor-core head
    groups only): False / 0 atomic adds, True / 1 per-slot dQ partials summed in slot order, 2 one dQ
    accumulator whose adds per token go in decreasing block order (ATTN_DQ_ORDERED); grad_fp32 makes dq, dk, dv fp32; atten_mask (attenMaskOptional) is a 2-D uint8 CUDA
    tensor [rows, cols] over local (query, key) positions, nonzero = key removed, covering every
    sequence (held by the descriptor)."""
    keep = _Keep()
    if atten_mask is not None:
        if atten_mask.dim() != 2 or not atten_mask.is_contiguous() or atten_mask.element_size() != 1:
            raise ValueError("atten_mask: a contiguous 2-D tensor of 1-byte elements")
        keep.items.append(atten_mask)
    desc = attn_nsa_desc_t(int(dtype), len(cu_seqlens_q), _cu_array(keep, cu_seqlens_q),
                           _cu_array(keep, cu_seqlens_kv), int(n1), int(n2), int(d), float(scale),
                           int(block_size), int(block_count), int(sparse_mode), int(deterministic),
                           int(d_v), int(bool(grad_fp32)),
                           atten_mask.data_ptr() if atten_mask is not None else None,
                           int(atten_mask.shape[0]) if atten_mask is not None else 0,
                           int(atten_mask.shape[1]) if atten_mask is not None else 0)
    desc._keep = keep
    return desc


def view_bhsd(t) -> attn_view_t:
    """A [B, H, S, D] tensor (any strides, innermost 1) as an attn_view_t."""
    if t.dim() != 4 or (t.shape[-1] > 1 and t.stride(-1) != 1):
        raise ValueError("expected a [B,H,S,D] tensor with unit innermost stride")
    sb, sh, ss, _ = t.stride()
    return attn_view_t(t.data_ptr(), sb, sh, ss)


def view_tnd(t) -> attn_view_t:
    """A packed [T, H, D] tensor as an attn_view_t (token stride = ss)."""
    if t.dim() != 3 or (t.shape[-1] > 1 and t.stride(-1) != 1):
        raise ValueError("expected a [T,H,D] tensor with unit innermost stride")
    st, sh, _ = t.stride()
    return attn_view_t(t.data_ptr(), 0, sh, st)


def sdpa_workspace_size(desc):
    """(forward bytes, backward bytes) of device workspace for this descriptor (host only)."""
    fwd, bwd = C.c_size_t(), C.c_size_t()
    check(_lib.load().sdpa_workspace_size(C.byref(desc), C.byref(fwd), C.byref(bwd)), "sdpa_workspace_size")
    return fwd.value, bwd.value


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def sdpa_fwd_stats(desc, q, k, v, o, lse, *, workspace=None, stream=None):
    """q, k, v, o: views (attn_view_t) or tensors; lse: fp32 CUDA tensor."""
    fwd, _ = sdpa_workspace_size(desc)
    ws = _workspace(fwd, lse.device, workspace)
    vq, vk, vv, vo = (x if isinstance(x, attn_view_t) else view_bhsd(x) for x in (q, k, v, o))
    st = _lib.load().sdpa_fwd_stats(C.byref(desc), vq, vk, vv, vo,
                                    C.cast(C.c_void_p(lse.data_ptr()), C.POINTER(C.c_float)),
                                    C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel()), C.c_void_p(_stream_ptr(stream)))
    check(st, "sdpa_fwd_stats")
    return ws


def sdpa_bwd(desc, q, k, v, o, dO, lse, dQ, dK, dV, *, workspace=None, stream=None):
    """dQ, dK, dV of scaled dot-product attention from O, dO and the fp32 stats lse (as sdpa_fwd_stats
    writes them).  Tensors are attn_view_t views or [B, H, S, D] CUDA tensors (view_bhsd); the call is
    asynchronous on `stream` (default: the current stream).  A workspace of the size
    sdpa_workspace_size gives is allocated when none is passed; it is returned, for attn_query_status."""
    _, bwd = sdpa_workspace_size(desc)
    ws = _workspace(bwd, lse.device, workspace)
    views = [x if isinstance(x, attn_view_t) else view_bhsd(x) for x in (q, k, v, o, dO, dQ, dK, dV)]
    st = _lib.load().sdpa_bwd(C.byref(desc), *views[:5],
                              C.cast(C.c_void_p(lse.data_ptr()), C.POINTER(C.c_float)), *views[5:],
                              C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel()), C.c_void_p(_stream_ptr(stream)))
    check(st, "sdpa_bwd")
    return ws


def nsa_workspace_size(desc):
    """Bytes of device workspace nsa_selected_attn_bwd needs for this descriptor (host only)."""
    n = C.c_size_t()
    check(_lib.load().nsa_workspace_size(C.byref(desc), C.byref(n)), "nsa_workspace_size")
    return n.value


def nsa_selected_attn_bwd(desc, q, k, v, o, dO, softmax_max, softmax_sum, topk, dq, dk, dv, *, workspace=None,
                          stream=None):
    """NSA selected-attention backward on contiguous TND CUDA tensors: q, o, dO, dq [T1, n1, d]; k, v,
    dk, dv [T2, n2, d]; softmax_max / softmax_sum [T1, n1, 8] fp32; topk [T1, n2, block_count] int32.
    Asynchronous on `stream`; returns the workspace (allocated when none is passed) for
    attn_query_status, which reports indices that were out of range or repeated."""
    ws = _workspace(nsa_workspace_size(desc), q.device, workspace)
    fp = lambda t: C.cast(C.c_void_p(t.data_ptr()), C.POINTER(C.c_float))
    st = _lib.load().nsa_selected_attn_bwd(
        C.byref(desc), *(C.c_void_p(t.data_ptr()) for t in (q, k, v, o, dO)), fp(softmax_max), fp(softmax_sum),
        C.cast(C.c_void_p(topk.data_ptr()), C.POINTER(C.c_int32)),
        *(C.c_void_p(t.data_ptr()) for t in (dq, dk, dv)), C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel()),
        C.c_void_p(_stream_ptr(stream)))
    check(st, "nsa_selected_attn_bwd")
    return ws


def nsa_fwd_workspace_size(desc):
    """Bytes of device workspace nsa_selected_attn_fwd needs (host only)."""
    n = C.c_size_t()
    check(_lib.load().nsa_fwd_workspace_size(C.byref(desc), C.byref(n)), "nsa_fwd_workspace_size")
    return n.value


def nsa_selected_attn_fwd(desc, q, k, v, topk, o, softmax_max, softmax_sum, *, workspace=None, stream=None):
    """NSA selected-attention forward on contiguous TND CUDA tensors: q [T1, n1, d], k [T2, n2, d],
    v [T2, n2, d_v], topk [T1, n2, block_count] int32 -> o [T1, n1, d_v] (input dtype), softmax_max /
    softmax_sum [T1, n1, 8] fp32.  Asynchronous on `stream`; returns the workspace (its first word is the
    device status)."""
    ws = _workspace(nsa_fwd_workspace_size(desc), q.device, workspace)
    fp = lambda t: C.cast(C.c_void_p(t.data_ptr()), C.POINTER(C.c_float))
    st = _lib.load().nsa_selected_attn_fwd(
        C.byref(desc), *(C.c_void_p(t.data_ptr()) for t in (q, k, v)),
        C.cast(C.c_void_p(topk.data_ptr()), C.POINTER(C.c_int32)), C.c_void_p(o.data_ptr()), fp(softmax_max),
        fp(softmax_sum), C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel()), C.c_void_p(_stream_ptr(stream)))
    check(st, "nsa_selected_attn_fwd")
    return ws


def nsa_block_lists(desc, topk, offsets, tokens, *, workspace=None, stream=None):
    """Fills device int32 tensors offsets / tokens; returns nblk_max."""
    ws = _workspace(nsa_workspace_size(desc), topk.device, workspace)
    ip = lambda t: C.cast(C.c_void_p(t.data_ptr()), C.POINTER(C.c_int32))
    nblk = C.c_int64()
    st = _lib.load().nsa_block_lists(C.byref(desc), ip(topk), ip(offsets), ip(tokens), C.byref(nblk),
                                     C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel()),
                                     C.c_void_p(_stream_ptr(stream)))
    check(st, "nsa_block_lists")
    return nblk.value, ws


def attn_query_status(workspace, stream=None):
    """Synchronises the stream; returns the device status bits (0 = clean)."""
    flags = C.c_uint32()
    st = _lib.load().attn_query_status(C.c_void_p(workspace.data_ptr()), C.c_void_p(_stream_ptr(stream)),
                                       C.byref(flags))
    if st not in (_lib.ATTN_OK, _lib.ATTN_ERR_DEVICE):
        check(st, "attn_query_status")
    return flags.value
