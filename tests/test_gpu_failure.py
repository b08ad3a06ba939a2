"""The device failure path on a GPU, without faulting it: a bounded mbarrier
wait that nothing completes runs out after a short limit, the kernel sets
ATTN_DEV_TIMEOUT in the workspace status word and returns, the host reads the
flag back, and the context stays usable for the next call."""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_flag_and_context_survives():
    import torch
    import attention_backward_02_gb300 as ab
    lib = ab._lib.load()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.attn_selftest_wait_timeout(C.c_void_p(ws.data_ptr()), C.c_size_t(256), C.c_double(0.02),
                                        C.c_void_p(stream))
    ab.check(st, "attn_selftest_wait_timeout")
    assert ab.attn_query_status(ws) == ab._lib.ATTN_DEV_TIMEOUT
    assert ab.attn_query_status(ws) == 0  # read and cleared
    # the context still runs the backward correctly
    p = synth.dense_problem("after_timeout", dtype=synth.F16, b=1, h=2, h_kv=2, d=64, s_q=200, s_kv=200,
                            mask=oracle.CAUSAL_TOP_LEFT, seed=41)
    o_bits, lse = H.oracle_forward(p)
    dq, dk, dv = H.run_gpu_bwd(p, o_bits, lse)
    rq, rk, rv = oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                                  p.f64("do"), lse, p.cu_q, p.cu_kv, p.scale, p.mask)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")
    assert np.all(np.isfinite(dq))


@pytest.mark.parametrize("mode", [0, 2])
def test_backward_while_other_work_holds_some_sms(mode):
    """While another stream's kernel holds 8 SMs (and their shared memory) for 1.5 s, longer than any
    wait's one-second limit, the backward must still complete correctly.  Atomic dQ mode: no block
    waits for another.  Ordered dQ mode: blocks wait for other blocks' adds, so the launch is
    cooperative and its blocks run only once they can all be resident."""
    import torch
    import attention_backward_02_gb300 as ab
    lib = ab._lib.load()
    p = synth.dense_problem("shared_gpu", dtype=synth.F16, b=1, h=16, h_kv=16, d=64, s_q=1280, s_kv=1280,
                            scale=0.125, mask=oracle.CAUSAL_TOP_LEFT, seed=43)  # 160 work units >= the SMs
    o_bits, lse = H.oracle_forward(p)
    ref = oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype), p.f64("do"),
                           lse, p.cu_q, p.cu_kv, p.scale, p.mask)
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    ab.check(lib.attn_selftest_occupy(8, 120 * 1024, C.c_double(1.5), C.c_void_p(other.cuda_stream)),
             "attn_selftest_occupy")
    dq, dk, dv = H.run_gpu_bwd(p, o_bits, lse, deterministic=mode)  # asserts a clean device status
    torch.cuda.synchronize()
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        H.assert_close(g, r, name)


@pytest.mark.parametrize("mode", [False, 2])
def test_nsa_backward_while_other_work_holds_some_sms(mode):
    """The NSA backward beside a kernel that holds 8 SMs for 1.5 s: atomic dQ (no block waits for another)
    and the ordered deterministic mode (blocks wait for other blocks' adds; a cooperative launch) both
    complete with oracle parity and a clean status."""
    import torch
    import attention_backward_02_gb300 as ab
    lib = ab._lib.load()
    p = synth.nsa_problem("shared_gpu_nsa", dtype=synth.BF16, lens_q=[1024, 700], lens_kv=[1024, 768], n1=16,
                          n2=2, d=128, block_size=64, block_count=6, sparse_mode=2, seed=44)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    ref = oracle.nsa_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype), p.f64("do"),
                         mx.astype(np.float64), sm.astype(np.float64), p.topk, p.cu_q, p.cu_kv, p.scale,
                         p.block_size, p.sparse_mode)
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    ab.check(lib.attn_selftest_occupy(8, 120 * 1024, C.c_double(1.5), C.c_void_p(other.cuda_stream)),
             "attn_selftest_occupy")
    got = H.run_gpu_nsa(p, o_bits, mx, sm, mode)  # asserts a clean device status
    torch.cuda.synchronize()
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        H.assert_close(g, r, name)
