"""The C ABI calls inside a CUDA graph: sdpa_bwd and sdpa_fwd_stats are
asynchronous on the caller's stream, allocate nothing and never synchronise,
so a captured call replays to the results of a direct call.  Expected values
come from the direct call (bitwise, in the deterministic dQ modes and for the
forward) and from the oracle (within the tolerance)."""
import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _setup(p, deterministic):
    import torch
    import attention_backward_02_gb300 as ab
    q, k, v, do = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do))
    o_bits, lse_td = H.oracle_forward(p)
    o = H.bits_to_gpu(o_bits, p.dtype)
    lse = torch.from_numpy(H.lse_layout(p, lse_td).astype(np.float32)).cuda()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    desc = H.dense_desc(p, deterministic)
    ws = torch.empty(ab.sdpa_workspace_size(desc)[1], dtype=torch.uint8, device="cuda")
    views = H.dense_views(p, (q, k, v, o, do, dq, dk, dv))
    keep = (q, k, v, o, do)  # the views hold raw pointers: the tensors must outlive them
    return desc, views, lse, ws, (dq, dk, dv), o_bits, lse_td, keep


@pytest.mark.parametrize("deterministic", [True, False, 2])
def test_backward_replayed_from_a_cuda_graph(deterministic):
    """Split, atomic and ordered dQ (the ordered mode's cooperative launch becomes a graph node too)."""
    import torch
    import attention_backward_02_gb300 as ab
    p = synth.dense_problem("graph", dtype=synth.F16, b=2, h=4, h_kv=2, d=64, s_q=300, s_kv=300,
                            mask=oracle.CAUSAL_TOP_LEFT, scale=0.125, seed=61)
    desc, (vq, vk, vv, vo, vdo, vdq, vdk, vdv), lse, ws, outs, o_bits, lse_td, _keep = _setup(p, deterministic)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        ab.sdpa_bwd(desc, vq, vk, vv, vo, vdo, lse, vdq, vdk, vdv, workspace=ws)  # direct call
    torch.cuda.synchronize()
    direct = [H.gpu_to_f64(t) for t in outs]
    assert ab.attn_query_status(ws) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ab.sdpa_bwd(desc, vq, vk, vv, vo, vdo, lse, vdq, vdk, vdv, workspace=ws)
    for t in outs:
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert ab.attn_query_status(ws) == 0
    replayed = [H.gpu_to_f64(t) for t in outs]
    ref = oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype), p.f64("do"),
                           lse_td, p.cu_q, p.cu_kv, p.scale, p.mask)
    for name, a, b, r in zip(("dQ", "dK", "dV"), direct, replayed, ref):
        if deterministic:  # split or ordered: the same bits
            np.testing.assert_array_equal(a, b)
        H.assert_close(b, r, name)


def test_forward_replayed_from_a_cuda_graph():
    import torch
    import attention_backward_02_gb300 as ab
    p = synth.dense_problem("graph_fwd", dtype=synth.BF16, b=2, h=4, h_kv=2, d=128, s_q=200, s_kv=333,
                            mask=oracle.CAUSAL_BOTTOM_RIGHT, seed=62)
    q, k, v = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v))
    o = torch.empty_like(q)
    lse = torch.empty(p.t_q * p.h, dtype=torch.float32, device="cuda")
    desc = H.dense_desc(p)
    vq, vk, vv, vo = H.dense_views(p, (q, k, v, o))
    ws = torch.empty(ab.sdpa_workspace_size(desc)[0], dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        ab.sdpa_fwd_stats(desc, vq, vk, vv, vo, lse, workspace=ws)
    torch.cuda.synchronize()
    o_direct, lse_direct = H.gpu_to_f64(o), lse.cpu().numpy().copy()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ab.sdpa_fwd_stats(desc, vq, vk, vv, vo, lse, workspace=ws)
    o.fill_(float("nan"))
    lse.fill_(float("nan"))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(H.gpu_to_f64(o), o_direct)  # one writer per element: the same bits
    np.testing.assert_array_equal(lse.cpu().numpy(), lse_direct)


@pytest.mark.parametrize("mode", [False, True, 2])
def test_nsa_backward_replayed_from_a_cuda_graph(mode):
    """nsa_selected_attn_bwd captured in a CUDA graph (the ordered mode's cooperative launch becomes a graph
    node too): the replay gives the direct call's bits in the deterministic modes and oracle parity in all."""
    import torch
    import attention_backward_02_gb300 as ab
    p = synth.nsa_problem("graph_nsa", dtype=synth.BF16, lens_q=[300, 129], lens_kv=[512, 256], n1=16, n2=2,
                          d=128, block_size=64, block_count=4, sparse_mode=2, seed=63)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    q, k, v, do, o = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do, o_bits))
    mx8 = torch.from_numpy(np.repeat(mx[..., None], 8, -1).astype(np.float32)).cuda()
    sm8 = torch.from_numpy(np.repeat(sm[..., None], 8, -1).astype(np.float32)).cuda()
    tk = torch.from_numpy(np.ascontiguousarray(p.topk, np.int32)).cuda()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    desc = H.nsa_desc(p, mode)
    ws = torch.empty(ab.nsa_workspace_size(desc), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        ab.nsa_selected_attn_bwd(desc, q, k, v, o, do, mx8, sm8, tk, dq, dk, dv, workspace=ws)
    torch.cuda.synchronize()
    direct = [H.gpu_to_f64(t) for t in (dq, dk, dv)]
    assert ab.attn_query_status(ws) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ab.nsa_selected_attn_bwd(desc, q, k, v, o, do, mx8, sm8, tk, dq, dk, dv, workspace=ws)
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert ab.attn_query_status(ws) == 0
    replayed = [H.gpu_to_f64(t) for t in (dq, dk, dv)]
    ref = oracle.nsa_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype), p.f64("do"),
                         mx.astype(np.float64), sm.astype(np.float64), p.topk, p.cu_q, p.cu_kv, p.scale,
                         p.block_size, p.sparse_mode)
    for name, a, b, r in zip(("dQ", "dK", "dV"), direct, replayed, ref):
        if mode:
            np.testing.assert_array_equal(a, b)
        H.assert_close(b, r, name)
