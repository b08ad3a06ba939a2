"""sdpa_bwd_static_scratch: the allocation-free variant of sdpa_bwd.

It exists for callers that cannot allocate device memory when they run the
backward (engines or plugins that own all device memory, loops that must not
allocate once running); it uses a scratch array compiled into the library
instead of a caller workspace.  Its results must match sdpa_bwd's on the same
inputs, call after call, whatever an earlier call left in the shared scratch.

Kept in a file that sorts last so that a run stopping at the first failure
has run every other test before this one.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ab():
    from attention_backward_02_gb300 import build
    build.build()
    import attention_backward_02_gb300 as ab
    ab._lib.load()
    return ab


def _static_status(ab):
    """Device status flags of the static scratch after the last call (read and cleared)."""
    import torch
    flags = C.c_uint32()
    st = ab._lib.load().attn_static_scratch_status(C.c_void_p(torch.cuda.current_stream().cuda_stream),
                                                  C.byref(flags))
    assert st in (ab._lib.ATTN_OK, ab._lib.ATTN_ERR_DEVICE), st
    return flags.value


def _static_call(ab, p, o_bits, lse_td, deterministic=False):
    import torch
    q, k, v, do, o = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do, o_bits))
    lse = torch.from_numpy(H.lse_layout(p, lse_td).astype(np.float32)).cuda()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    desc = H.dense_desc(p, deterministic)
    views = H.dense_views(p, (q, k, v, o, do, dq, dk, dv))
    stream = torch.cuda.current_stream().cuda_stream
    st = ab._lib.load().sdpa_bwd_static_scratch(C.byref(desc), *views[:5],
                                                C.cast(C.c_void_p(lse.data_ptr()), C.POINTER(C.c_float)),
                                                *views[5:], C.c_void_p(stream))
    ab.check(st, "sdpa_bwd_static_scratch")
    torch.cuda.synchronize()
    return H.gpu_to_f64(dq), H.gpu_to_f64(dk), H.gpu_to_f64(dv)


def _oracle_bwd(p, o_bits, lse):
    return oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype), p.f64("do"),
                            lse, p.cu_q, p.cu_kv, p.scale, p.mask)


def test_static_scratch_matches_workspace_entry_point_twice(ab):
    problems = [
        (synth.dense_problem("noalloc_a", dtype=synth.F16, b=2, h=4, h_kv=4, d=64, s_q=256, s_kv=256,
                             scale=0.125, mask=1, seed=301), False),
        (synth.dense_problem("noalloc_b", dtype=synth.BF16, b=1, h=8, h_kv=2, d=128, s_q=200, s_kv=333,
                             mask=2, seed=302), False),
        # deterministic mode: split partial dQ buffers and the separate finalize kernel, in the scratch
        (synth.dense_problem("noalloc_c", dtype=synth.F16, b=1, h=4, h_kv=2, d=64, s_q=300, s_kv=300,
                             scale=0.125, mask=1, seed=303), True),
        # packed sequences, causal bottom-right: the workspace rows follow the sequence lengths
        (synth.dense_problem("noalloc_d", dtype=synth.BF16, b=3, h=4, h_kv=2, d=128,
                             lens_q=np.array([70, 200, 129]), lens_kv=np.array([90, 200, 140]), mask=2,
                             seed=304), False),
    ]
    for p, det in problems:  # calls in a row, different shapes and modes, one shared scratch
        o_bits, lse = H.oracle_forward(p)
        got = _static_call(ab, p, o_bits, lse, det)
        assert _static_status(ab) == 0
        ref = H.run_gpu_bwd(p, o_bits, lse, det)
        exact = _oracle_bwd(p, o_bits, lse)
        for name, g, r, x in zip(("dQ", "dK", "dV"), got, ref, exact):
            H.assert_close(g, x, f"{p.name} {name} vs oracle")
            H.assert_close(g, r, f"{p.name} {name} vs sdpa_bwd")
            if det:  # same kernels, same fixed order: the same bits
                np.testing.assert_array_equal(g, r)


def test_static_scratch_rejects_oversized_problem(ab):
    p_desc = ab.sdpa_desc(dtype=ab.ATTN_BF16, b=8, h=32, h_kv=32, s_q=4096, s_kv=4096, d=128, scale=0.088,
                          mask=ab.ATTN_CAUSAL_TOP_LEFT)
    _, need = ab.sdpa_workspace_size(p_desc)
    assert need > (16 << 20)
    v = ab.attn_view_t(0x10000, 0, 0, 0)
    st = ab._lib.load().sdpa_bwd_static_scratch(C.byref(p_desc), v, v, v, v, v,
                                                C.cast(C.c_void_p(0x20000), C.POINTER(C.c_float)), v, v, v, None)
    assert st == ab._lib.ATTN_ERR_WORKSPACE
