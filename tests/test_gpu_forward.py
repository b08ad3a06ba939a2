"""GPU parity of the dense SDPA forward (sdpa_fwd_stats: O and the fp32
log-sum-exp stats) against the fp64 oracle's forward, through the C ABI.
Expected values come only from the oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu

F16, BF16 = synth.F16, synth.BF16
NONE, TL, BR = oracle.MASK_NONE, oracle.CAUSAL_TOP_LEFT, oracle.CAUSAL_BOTTOM_RIGHT


def _fwd_parity(p, ro=None, rlse=None):
    o, lse = H.run_gpu_fwd(p)
    if ro is None:
        ro, rlse = oracle.dense_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.cu_q, p.cu_kv, p.scale, p.mask)
    H.assert_close(o, ro, "O")
    finite = np.isfinite(rlse)
    # rows that see no key: LSE = +inf and O = 0
    assert np.all(np.isposinf(lse[~finite])), "rows without keys must have LSE = +inf"
    np.testing.assert_allclose(lse[finite], rlse[finite], rtol=1e-5, atol=1e-5)
    return o, lse


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [NONE, TL, BR])
def test_forward_small_shapes(dtype, d, mask):
    """Several query and key tiles with ragged tails, s_q != s_kv, grouped-query heads."""
    p = synth.dense_problem("fwd_small", dtype=dtype, b=2, h=4, h_kv=2, d=d, s_q=200, s_kv=333, mask=mask,
                            seed=500 + d + mask + 7 * dtype)
    _fwd_parity(p)


@pytest.mark.parametrize("s_q,s_kv", [(1, 1), (300, 10), (129, 1), (10, 300)])
def test_forward_edge_lengths(s_q, s_kv):
    """Single rows, rows without keys under bottom-right alignment (s_q > s_kv), short key ranges."""
    p = synth.dense_problem("fwd_edge", dtype=F16, b=2, h=2, h_kv=1, d=64, s_q=s_q, s_kv=s_kv, mask=BR,
                            seed=510 + s_q + s_kv)
    _fwd_parity(p)


@pytest.mark.parametrize("d", [64, 128])
def test_forward_varlen_gqa(d):
    """Packed sequences (one empty, one without keys), grouped-query heads, causal bottom-right."""
    lq = np.array([1, 200, 0, 129, 77]); lkv = np.array([5, 150, 0, 0, 300])
    p = synth.dense_problem("fwd_varlen", dtype=BF16, b=len(lq), h=8, h_kv=2, d=d, lens_q=lq, lens_kv=lkv,
                            mask=BR, seed=520 + d)
    _fwd_parity(p)


def test_forward_large_scores():
    """Scores spread over a wide range (large scale): the running max is raised several times within a
    row, so the rescaling of O in TMEM is exercised."""
    p = synth.dense_problem("fwd_wide", dtype=BF16, b=1, h=2, h_kv=2, d=128, s_q=256, s_kv=1024, scale=1.0,
                            mask=NONE, seed=530)
    _fwd_parity(p)


def test_forward_workload1():
    """fp16 b4 h12 s1024 d64 causal, BSHD viewed as BHSD: every O element and stat."""
    _fwd_parity(synth.workload(1))


@pytest.mark.slow
@pytest.mark.parametrize("idx", [2, 3])
def test_forward_workloads_2_3(idx):
    """bf16 b2 h32 s4096 d128 causal; varlen GQA 32/8 d128 causal bottom-right: every element."""
    p = synth.workload(idx)
    ro, rlse = oracle.dense_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.cu_q, p.cu_kv, p.scale, p.mask)
    _fwd_parity(p, ro, rlse)
