"""fp64 CPU oracle for SDPA forward/backward and NSA selected-attention backward.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports, links
or calls anything here, and nothing here imports the CUDA library.

This module is a thin ctypes wrapper over ``attn_oracle.c`` (the definitions,
with their citations, live in that file's header).  All arrays are numpy
float64 in token-major (TND) layout:

    q, o, do, dq : [Tq, h, d]     k, v, dk, dv : [Tkv, h_kv, d]
    lse, max, sum: [Tq, h]        topk         : [Tq, h_kv, cnt] int32

Sequences are inclusive cumulative lengths without a leading zero (the form
of the Ascend page's actualSeqQLen / actualSeqKvLen).  In the NSA functions
value, O and dO may have a head dim of their own (the page allows the value
head dim to differ from the query / key one); it is read off v's shape.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

MASK_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable C11 + pthreads)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-D_POSIX_C_SOURCE=200809L",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dense(C.Structure):
    _fields_ = [("nseq", C.c_int64), ("cu_q", C.POINTER(C.c_int64)), ("cu_kv", C.POINTER(C.c_int64)),
                ("h", C.c_int64), ("h_kv", C.c_int64), ("d", C.c_int64), ("scale", C.c_double),
                ("mask", C.c_int)]


class _Nsa(C.Structure):
    _fields_ = [("nseq", C.c_int64), ("cu_q", C.POINTER(C.c_int64)), ("cu_kv", C.POINTER(C.c_int64)),
                ("n1", C.c_int64), ("n2", C.c_int64), ("d", C.c_int64), ("scale", C.c_double),
                ("block_size", C.c_int64), ("block_count", C.c_int64), ("sparse_mode", C.c_int),
                ("d_v", C.c_int64), ("atten_mask", C.POINTER(C.c_uint8)), ("mask_rows", C.c_int64),
                ("mask_cols", C.c_int64)]


def _load():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
    return _lib


def thread_count() -> int:
    """Threads the oracle uses by default (ORACLE_THREADS, else online cores)."""
    return int(_load().ora_thread_count())


def _d(a):
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _cu(cu):
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int64))


def _dense_desc(cu_q, cu_kv, h, h_kv, d, scale, mask):
    desc = _Dense(len(cu_q), cu_q.ctypes.data_as(C.POINTER(C.c_int64)),
                  cu_kv.ctypes.data_as(C.POINTER(C.c_int64)), h, h_kv, d, float(scale), int(mask))
    return desc


def dense_fwd(q, k, v, cu_q, cu_kv, scale, mask=MASK_NONE, threads=0):
    """O [Tq,h,d] and natural-log LSE [Tq,h] of the scaled, masked scores."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    tq, h, d = q.shape
    h_kv = k.shape[1]
    o = np.empty_like(q)
    lse = np.empty((tq, h), np.float64)
    desc = _dense_desc(cu_q, cu_kv, h, h_kv, d, scale, mask)
    rc = _load().ora_dense_fwd(C.byref(desc), _d(q), _d(k), _d(v), _d(o), _d(lse), int(threads))
    if rc:
        raise ValueError("oracle dense_fwd rejected its arguments")
    return o, lse


def dense_bwd(q, k, v, o, do, lse, cu_q, cu_kv, scale, mask=MASK_NONE, threads=0):
    """dQ, dK, dV with D computed from the supplied O and P from the supplied LSE."""
    q, k, v, o, do, lse = (_f64(x) for x in (q, k, v, o, do, lse))
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    tq, h, d = q.shape
    h_kv = k.shape[1]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    desc = _dense_desc(cu_q, cu_kv, h, h_kv, d, scale, mask)
    rc = _load().ora_dense_bwd(C.byref(desc), _d(q), _d(k), _d(v), _d(o), _d(do), _d(lse),
                               _d(dq), _d(dk), _d(dv), int(threads))
    if rc:
        raise ValueError("oracle dense_bwd rejected its arguments")
    return dq, dk, dv


def dense_bwd_rows(q, k, v, o, do, lse, cu_q, cu_kv, scale, mask, q_rows, kv_rows, threads=0):
    """The backward evaluated only at chosen rows.

    q_rows  : int64 array of token*h + head     -> dq rows  [len, d]
    kv_rows : int64 array of token*h_kv + head  -> dk, dv rows [len, d]
    """
    q, k, v, o, do, lse = (_f64(x) for x in (q, k, v, o, do, lse))
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    _, h, d = q.shape
    h_kv = k.shape[1]
    q_rows = np.ascontiguousarray(q_rows, np.int64)
    kv_rows = np.ascontiguousarray(kv_rows, np.int64)
    dq = np.empty((len(q_rows), d)); dk = np.empty((len(kv_rows), d)); dv = np.empty((len(kv_rows), d))
    desc = _dense_desc(cu_q, cu_kv, h, h_kv, d, scale, mask)
    p64 = lambda a: a.ctypes.data_as(C.POINTER(C.c_int64))
    rc = _load().ora_dense_bwd_rows(C.byref(desc), _d(q), _d(k), _d(v), _d(o), _d(do), _d(lse),
                                    C.c_int64(len(q_rows)), p64(q_rows), _d(dq),
                                    C.c_int64(len(kv_rows)), p64(kv_rows), _d(dk), _d(dv), int(threads))
    if rc:
        raise ValueError("oracle dense_bwd_rows rejected its arguments")
    return dq, dk, dv


def _mask(mask):
    """attenMaskOptional as a C-contiguous uint8 [rows, cols] array (nonzero: key removed), or None."""
    if mask is None:
        return None
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    if m.ndim != 2:
        raise ValueError("attenMaskOptional is 2-D: [query positions, key positions]")
    return m


def _nsa_desc(cu_q, cu_kv, n1, n2, d, scale, bs, cnt, sparse_mode, d_v=0, mask=None):
    """mask: the uint8 array from _mask (kept alive by the caller) or None."""
    mp = mask.ctypes.data_as(C.POINTER(C.c_uint8)) if mask is not None else None
    rows, cols = (mask.shape if mask is not None else (0, 0))
    return _Nsa(len(cu_q), cu_q.ctypes.data_as(C.POINTER(C.c_int64)),
                cu_kv.ctypes.data_as(C.POINTER(C.c_int64)), n1, n2, d, float(scale), bs, cnt,
                int(sparse_mode), int(d_v), mp, int(rows), int(cols))


def _nsa_dims(q, k, v):
    """(d, d_v): query / key head dim and value head dim (the Ascend page lets them differ)."""
    if k.shape[2] != q.shape[2]:
        raise ValueError("query and key head dims differ")
    return q.shape[2], v.shape[2]


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _ip(a):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


def nsa_fwd(q, k, v, topk, cu_q, cu_kv, scale, block_size, sparse_mode, threads=0, mask=None):
    """Sparse forward: O [T1,n1,d], softmaxMax [T1,n1], softmaxSum [T1,n1].  mask: optional 2-D
    attenMaskOptional over (query, key) positions local to the sequence, nonzero = removed."""
    q, k, v, topk = _f64(q), _f64(k), _f64(v), _i32(topk)
    mask = _mask(mask)
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    t1, n1, _ = q.shape
    d, dv_ = _nsa_dims(q, k, v)
    n2, cnt = k.shape[1], topk.shape[2]
    o = np.empty((t1, n1, dv_)); mx = np.empty((t1, n1)); sm = np.empty((t1, n1))
    desc = _nsa_desc(cu_q, cu_kv, n1, n2, d, scale, block_size, cnt, sparse_mode, dv_, mask)
    rc = _load().ora_nsa_fwd(C.byref(desc), _d(q), _d(k), _d(v), _ip(topk), _d(o), _d(mx), _d(sm),
                             int(threads))
    if rc:
        raise ValueError("oracle nsa_fwd rejected its arguments or an index")
    return o, mx, sm


def nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, scale, block_size, sparse_mode, threads=0, mask=None):
    """Gather -> dense backward on the gathered rows -> scatter-add back.  mask as for nsa_fwd."""
    q, k, v, o, do, mx, sm = (_f64(x) for x in (q, k, v, o, do, mx, sm))
    mask = _mask(mask)
    topk = _i32(topk)
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    _, n1, _ = q.shape
    d, dv_ = _nsa_dims(q, k, v)
    if o.shape[2] != dv_ or do.shape[2] != dv_:
        raise ValueError("attentionOut and its gradient must have the value head dim")
    n2, cnt = k.shape[1], topk.shape[2]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    desc = _nsa_desc(cu_q, cu_kv, n1, n2, d, scale, block_size, cnt, sparse_mode, dv_, mask)
    rc = _load().ora_nsa_bwd(C.byref(desc), _d(q), _d(k), _d(v), _d(o), _d(do), _d(mx), _d(sm),
                             _ip(topk), _d(dq), _d(dk), _d(dv), int(threads))
    if rc:
        raise ValueError("oracle nsa_bwd rejected its arguments or an index")
    return dq, dk, dv


def nsa_masked_dense(q, k, v, do, topk, cu_q, cu_kv, scale, block_size, sparse_mode, threads=0, mask=None):
    """Independent NSA path: masked dense attention, own softmax; returns o, dq, dk, dv."""
    q, k, v, do, topk = _f64(q), _f64(k), _f64(v), _f64(do), _i32(topk)
    mask = _mask(mask)
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    t1, n1, _ = q.shape
    d, dv_ = _nsa_dims(q, k, v)
    if do.shape[2] != dv_:
        raise ValueError("the gradient of attentionOut must have the value head dim")
    n2, cnt = k.shape[1], topk.shape[2]
    o, dq, dk, dv = np.empty((t1, n1, dv_)), np.empty_like(q), np.empty_like(k), np.empty_like(v)
    desc = _nsa_desc(cu_q, cu_kv, n1, n2, d, scale, block_size, cnt, sparse_mode, dv_, mask)
    rc = _load().ora_nsa_masked_dense(C.byref(desc), _d(q), _d(k), _d(v), _d(do), _ip(topk),
                                      _d(o), _d(dq), _d(dk), _d(dv), int(threads))
    if rc:
        raise ValueError("oracle nsa_masked_dense rejected its arguments or an index")
    return o, dq, dk, dv


def nsa_block_lists(topk, cu_q, cu_kv, n1, block_size, sparse_mode):
    """Per (sequence, kv head, block): ascending global ids of the tokens that
    selected the block and see at least one of its keys.  Returns (offsets,
    tokens, nblk_max) with offsets of length nseq*n2*nblk_max + 1."""
    topk = _i32(topk)
    cu_q, cu_kv = _cu(cu_q), _cu(cu_kv)
    t1, n2, cnt = topk.shape
    starts = np.concatenate([[0], cu_kv[:-1]])
    nblk_max = int(((cu_kv - starts) // block_size).max())
    offsets = np.zeros(len(cu_q) * n2 * nblk_max + 1, np.int64)
    tokens = np.zeros(max(1, t1 * n2 * cnt), np.int32)
    desc = _nsa_desc(cu_q, cu_kv, n1, n2, 1, 1.0, block_size, cnt, sparse_mode)
    rc = _load().ora_nsa_block_lists(C.byref(desc), _ip(topk), C.c_int64(nblk_max),
                                     offsets.ctypes.data_as(C.POINTER(C.c_int64)), _ip(tokens))
    if rc:
        raise ValueError("oracle nsa_block_lists rejected its arguments")
    return offsets, tokens[: offsets[-1]].copy(), nblk_max
