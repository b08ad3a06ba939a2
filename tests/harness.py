"""Shared test helpers: tolerance checks and marshalling of synthetic problems
onto the GPU through the C ABI.  Expected values come only from the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# Acceptance bar for fp16/bf16 inputs drawn from N(0,1): relative L2 error
# and an elementwise bound, both against the fp64 oracle.
REL_L2 = 5e-3
ATOL = 2e-2
RTOL = 2e-2


def rel_l2(got, ref):
    """Relative L2 error.  The denominator is floored at the elementwise
    absolute tolerance scale (ATOL * sqrt(n)): where the exact gradient is
    (near) zero, e.g. a single key makes dS = 0, relative error is undefined
    and the elementwise bound alone decides."""
    floor = ATOL * np.sqrt(max(1, np.size(ref)))
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), floor))


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_l2(got, ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = np.abs(got - ref) > bound
    assert r <= REL_L2, f"{what}: relative L2 {r:.3e} > {REL_L2}"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond {ATOL} + {RTOL}|ref|, worst "
                           f"{float(np.max(np.abs(got - ref) - bound)):.3e}")
    return r


def oracle_forward(p: synth.DenseProblem, threads=0):
    """O rounded to the problem's 16-bit type, and fp64 LSE [T, h]."""
    o, lse = oracle.dense_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.cu_q, p.cu_kv, p.scale, p.mask,
                              threads=threads)
    o_bits = synth.to_bits(o.astype(np.float32), p.dtype)
    return o_bits, lse


# ------------------------------------------------------------------ GPU side

def torch_dtype(dtype):
    import torch
    return torch.float16 if dtype == synth.F16 else torch.bfloat16


def bits_to_gpu(bits, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch_dtype(dtype))


def gpu_to_f64(t):
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64)


def lse_layout(p: synth.DenseProblem, lse_td):
    """[T, h] -> the ABI layout: [B][h][s_q] fixed, [h][T] packed."""
    if p.varlen:
        return np.ascontiguousarray(lse_td.T)
    b, s = p.b, p.s_q
    return np.ascontiguousarray(lse_td.reshape(b, s, p.h).transpose(0, 2, 1))


def dense_views(p: synth.DenseProblem, tensors):
    """token-major [T, H, D] GPU tensors -> attn_view_t (BHSD over BSHD, or TND)."""
    import attention_backward_02_gb300 as ab
    out = []
    for t in tensors:
        if p.varlen:
            out.append(ab.view_tnd(t))
        else:
            s = t.shape[0] // p.b
            out.append(ab.view_bhsd(t.view(p.b, s, t.shape[1], t.shape[2]).permute(0, 2, 1, 3)))
    return out


def dense_desc(p: synth.DenseProblem, deterministic=False, dq_splits=0):
    import attention_backward_02_gb300 as ab
    kw = dict(dtype=p.dtype, b=p.b, h=p.h, h_kv=p.h_kv, d=p.d, scale=p.scale, mask=p.mask,
              deterministic=deterministic, dq_splits=dq_splits)
    if p.varlen:
        return ab.sdpa_desc(s_q=0, s_kv=0, cu_seqlens_q=list(p.cu_q), cu_seqlens_kv=list(p.cu_kv), **kw)
    return ab.sdpa_desc(s_q=p.s_q, s_kv=p.s_kv, **kw)


def run_gpu_bwd(p: synth.DenseProblem, o_bits, lse_td, deterministic=False, dq_splits=0, check_status=True):
    """Runs sdpa_bwd on the GPU; returns dq, dk, dv as fp64 [T, H, D]."""
    import torch
    import attention_backward_02_gb300 as ab
    q, k, v, do, o = (bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do, o_bits))
    lse = torch.from_numpy(lse_layout(p, lse_td).astype(np.float32)).cuda()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dq.fill_(float("nan")); dk.fill_(float("nan")); dv.fill_(float("nan"))
    desc = dense_desc(p, deterministic, dq_splits)
    vq, vk, vv, vo, vdo, vdq, vdk, vdv = dense_views(p, (q, k, v, o, do, dq, dk, dv))
    ws = ab.sdpa_bwd(desc, vq, vk, vv, vo, vdo, lse, vdq, vdk, vdv)
    if check_status:
        assert ab.attn_query_status(ws) == 0
    torch.cuda.synchronize()
    return gpu_to_f64(dq), gpu_to_f64(dk), gpu_to_f64(dv)


def run_gpu_fwd(p: synth.DenseProblem):
    """sdpa_fwd_stats on the GPU: O (16-bit bits as f64) [T,H,D] and LSE [T,H]."""
    import torch
    import attention_backward_02_gb300 as ab
    q, k, v = (bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v))
    o = torch.empty_like(q)
    n = p.t_q * p.h
    lse = torch.empty(n, dtype=torch.float32, device="cuda")
    desc = dense_desc(p)
    vq, vk, vv, vo = dense_views(p, (q, k, v, o))
    ab.sdpa_fwd_stats(desc, vq, vk, vv, vo, lse)
    torch.cuda.synchronize()
    lse = lse.cpu().numpy().astype(np.float64)
    if p.varlen:
        lse_td = lse.reshape(p.h, p.t_q).T
    else:
        lse_td = lse.reshape(p.b, p.h, p.s_q).transpose(0, 2, 1).reshape(p.t_q, p.h)
    return gpu_to_f64(o), lse_td


# ------------------------------------------------------------------------ NSA

def nsa_oracle_inputs(p: synth.NsaProblem, threads=0, mask=None):
    """Sparse forward by the oracle: O rounded to 16 bits, fp32 max / sum."""
    o, mx, sm = oracle.nsa_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.topk, p.cu_q, p.cu_kv, p.scale,
                               p.block_size, p.sparse_mode, threads=threads, mask=mask)
    o_bits = synth.to_bits(o.astype(np.float32), p.dtype)
    return o_bits, mx.astype(np.float32), sm.astype(np.float32)


def nsa_desc(p: synth.NsaProblem, deterministic=False, grad_fp32=False, mask=None):
    """mask: optional numpy 2-D attenMaskOptional (copied to the GPU; the descriptor holds it)."""
    import torch
    import attention_backward_02_gb300 as ab
    d_v = p.v.shape[-1]
    m = None if mask is None else torch.from_numpy(np.ascontiguousarray(mask != 0, dtype=np.uint8)).cuda()
    return ab.nsa_desc(dtype=p.dtype, cu_seqlens_q=list(p.cu_q), cu_seqlens_kv=list(p.cu_kv), n1=p.n1, n2=p.n2,
                       d=p.d, scale=p.scale, block_size=p.block_size, block_count=p.block_count,
                       sparse_mode=p.sparse_mode, deterministic=deterministic, d_v=0 if d_v == p.d else d_v,
                       grad_fp32=grad_fp32, atten_mask=m)


def run_gpu_nsa_fwd(p: synth.NsaProblem, topk=None, expect_flags=0, mask=None):
    """nsa_selected_attn_fwd on the GPU: O (16-bit values as f64), softmax max and sum (lane 0, f64)
    and the 8-lane stats as returned."""
    import torch
    import attention_backward_02_gb300 as ab
    q, k, v = (bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v))
    o = torch.full((p.t1, p.n1, p.v.shape[-1]), float("nan"), dtype=q.dtype, device="cuda")
    mx8 = torch.full((p.t1, p.n1, 8), float("nan"), dtype=torch.float32, device="cuda")
    sm8 = torch.full((p.t1, p.n1, 8), float("nan"), dtype=torch.float32, device="cuda")
    tk = torch.from_numpy(np.ascontiguousarray(p.topk if topk is None else topk, np.int32)).cuda()
    ws = ab.nsa_selected_attn_fwd(nsa_desc(p, mask=mask), q, k, v, tk, o, mx8, sm8)
    flags = ab.attn_query_status(ws)
    assert flags == expect_flags, f"device status {flags:#x}, expected {expect_flags:#x}"
    torch.cuda.synchronize()
    m8, s8 = mx8.cpu().numpy().astype(np.float64), sm8.cpu().numpy().astype(np.float64)
    return gpu_to_f64(o), m8[..., 0], s8[..., 0], m8, s8


def run_gpu_nsa(p: synth.NsaProblem, o_bits, mx, sm, deterministic=False, topk=None, expect_flags=0,
                grad_fp32=False, mask=None):
    import torch
    import attention_backward_02_gb300 as ab
    q, k, v, do, o = (bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do, o_bits))
    mx8 = torch.from_numpy(np.repeat(mx[..., None], 8, -1).astype(np.float32)).cuda()
    sm8 = torch.from_numpy(np.repeat(sm[..., None], 8, -1).astype(np.float32)).cuda()
    tk = torch.from_numpy(np.ascontiguousarray(p.topk if topk is None else topk, np.int32)).cuda()
    gdt = torch.float32 if grad_fp32 else q.dtype
    dq, dk, dv = (torch.empty(x.shape, dtype=gdt, device="cuda") for x in (q, k, v))
    dq.fill_(float("nan")); dk.fill_(float("nan")); dv.fill_(float("nan"))
    ws = ab.nsa_selected_attn_bwd(nsa_desc(p, deterministic, grad_fp32, mask), q, k, v, o, do, mx8, sm8, tk, dq,
                                  dk, dv)
    flags = ab.attn_query_status(ws)
    assert flags == expect_flags, f"device status {flags:#x}, expected {expect_flags:#x}"
    torch.cuda.synchronize()
    return gpu_to_f64(dq), gpu_to_f64(dk), gpu_to_f64(dv)
