"""GPU parity of the dense SDPA backward (and forward) against the fp64 oracle,
through the C ABI.  Expected values come only from the oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu

F16, BF16 = synth.F16, synth.BF16
NONE, TL, BR = oracle.MASK_NONE, oracle.CAUSAL_TOP_LEFT, oracle.CAUSAL_BOTTOM_RIGHT


def _parity(p, deterministic=False, dq_splits=0):
    o_bits, lse = H.oracle_forward(p)
    dq, dk, dv = H.run_gpu_bwd(p, o_bits, lse, deterministic, dq_splits)
    rq, rk, rv = oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                                  p.f64("do"), lse, p.cu_q, p.cu_kv, p.scale, p.mask)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")
    return dq, dk, dv


def test_workload0_forward_and_backward():
    """fp16 b1 h2 s128 d64, scale 1/8, non-causal: forward O/LSE and backward."""
    p = synth.workload(0)
    o, lse = H.run_gpu_fwd(p)
    ro, rlse = oracle.dense_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.cu_q, p.cu_kv, p.scale, p.mask)
    H.assert_close(o, ro, "O")
    np.testing.assert_allclose(lse, rlse, rtol=1e-5, atol=1e-5)
    _parity(p)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [NONE, TL, BR])
def test_small_shapes(dtype, d, mask):
    """Several tiles with ragged tails on both sides; s_q != s_kv for the masks."""
    p = synth.dense_problem("small", dtype=dtype, b=2, h=4, h_kv=2, d=d, s_q=200, s_kv=333, mask=mask,
                            seed=100 + d + mask)
    _parity(p)


@pytest.mark.parametrize("s_q,s_kv", [(1, 1), (1, 257), (129, 1), (64, 64), (300, 300)])
def test_edge_lengths(s_q, s_kv):
    p = synth.dense_problem("edge", dtype=BF16, b=1, h=2, h_kv=1, d=128, s_q=s_q, s_kv=s_kv, mask=BR,
                            seed=s_q * 7 + s_kv)
    _parity(p)


@pytest.mark.parametrize("s_q,s_kv", [(300, 10), (129, 1), (256, 300)])
def test_edge_lengths_d64(s_q, s_kv):
    """fp16, d = 64 (128-row query tiles): whole query tiles that no key reaches get dQ = 0 without
    any contribution being added for them."""
    p = synth.dense_problem("edge64", dtype=F16, b=2, h=2, h_kv=2, d=64, s_q=s_q, s_kv=s_kv, mask=BR,
                            seed=s_q * 5 + s_kv)
    _parity(p)


def test_varlen_gqa_small():
    lens = np.array([1, 130, 77, 256, 5, 300])
    p = synth.dense_problem("varlen", dtype=BF16, b=len(lens), h=8, h_kv=2, d=128, lens_q=lens, lens_kv=lens,
                            mask=BR, seed=7)
    _parity(p)


def test_varlen_unequal_lengths():
    lq = np.array([40, 200, 129]); lkv = np.array([100, 150, 129])
    p = synth.dense_problem("varlen2", dtype=F16, b=3, h=4, h_kv=4, d=64, lens_q=lq, lens_kv=lkv, mask=BR, seed=8)
    _parity(p)


def test_empty_sequence_in_batch():
    lens = np.array([64, 0, 100])
    p = synth.dense_problem("varlen0", dtype=BF16, b=3, h=2, h_kv=2, d=128, lens_q=lens, lens_kv=lens,
                            mask=TL, seed=9)
    _parity(p)


@pytest.mark.parametrize("d,mask", [(64, NONE), (64, BR), (128, BR)])
def test_sequence_without_keys(d, mask):
    """Varlen batch where one sequence has queries but no keys: its dQ rows are 0 (converted by the
    main kernel from the accumulator nothing was added to) and the other sequences are unaffected."""
    lq = np.array([64, 50, 100]); lkv = np.array([64, 0, 100])
    p = synth.dense_problem("nokeys", dtype=F16, b=3, h=2, h_kv=2, d=d, lens_q=lq, lens_kv=lkv, mask=mask,
                            seed=13 + d + mask)
    dq, _, _ = _parity(p)
    assert not np.any(dq[64:114])


def test_no_keys_at_all():
    """s_kv = 0: the main kernel has no work and does not run; the finalize writes dQ = 0."""
    p = synth.dense_problem("nokv", dtype=BF16, b=2, h=2, h_kv=1, d=64, s_q=70, s_kv=0, mask=NONE, seed=14)
    dq, dk, dv = _parity(p)
    assert not np.any(dq) and dk.size == 0 and dv.size == 0


@pytest.mark.parametrize("dq_splits", [0, 3])
def test_deterministic_mode_bitwise(dq_splits):
    p = synth.dense_problem("det", dtype=BF16, b=2, h=4, h_kv=2, d=128, s_q=520, s_kv=520, mask=TL, seed=11)
    o_bits, lse = H.oracle_forward(p)
    a = H.run_gpu_bwd(p, o_bits, lse, deterministic=True, dq_splits=dq_splits)
    b = H.run_gpu_bwd(p, o_bits, lse, deterministic=True, dq_splits=dq_splits)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    _parity(p, deterministic=True, dq_splits=dq_splits)


@pytest.mark.parametrize("dq_splits", [0, 2])
def test_deterministic_mode_bitwise_d64(dq_splits):
    """Deterministic mode at d = 64 (128-row query tiles, fp16), causal with ragged tails."""
    p = synth.dense_problem("det64", dtype=F16, b=2, h=4, h_kv=2, d=64, s_q=520, s_kv=520, mask=TL, scale=0.125,
                            seed=21)
    o_bits, lse = H.oracle_forward(p)
    a = H.run_gpu_bwd(p, o_bits, lse, deterministic=True, dq_splits=dq_splits)
    b = H.run_gpu_bwd(p, o_bits, lse, deterministic=True, dq_splits=dq_splits)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    _parity(p, deterministic=True, dq_splits=dq_splits)


ORDERED = 2  # ATTN_DQ_ORDERED


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [NONE, TL, BR])
def test_ordered_mode_bitwise(d, mask):
    """Ordered dQ mode (one fp32 buffer; each query tile's key tiles add in decreasing order behind a
    per-tile counter): oracle parity and the same bits from two calls, with s_q != s_kv, ragged
    tails, grouped-query heads and each mask."""
    p = synth.dense_problem("ord", dtype=BF16 if d == 128 else F16, b=2, h=4, h_kv=2, d=d, s_q=530, s_kv=700,
                            mask=mask, scale=1 / np.sqrt(d), seed=40 + d + mask)
    o_bits, lse = H.oracle_forward(p)
    a = H.run_gpu_bwd(p, o_bits, lse, deterministic=ORDERED)
    b = H.run_gpu_bwd(p, o_bits, lse, deterministic=ORDERED)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    _parity(p, deterministic=ORDERED)


@pytest.mark.parametrize("d", [64, 128])
def test_ordered_mode_varlen_gqa(d):
    """Ordered dQ mode with packed sequences of unequal lengths (one empty, one without keys),
    grouped-query heads, causal bottom-right."""
    lq = np.array([1, 200, 0, 129, 300, 77]); lkv = np.array([5, 150, 0, 0, 610, 400])
    p = synth.dense_problem("ord_varlen", dtype=BF16, b=len(lq), h=8, h_kv=2, d=d, lens_q=lq, lens_kv=lkv,
                            mask=BR, seed=50 + d)
    o_bits, lse = H.oracle_forward(p)
    a = H.run_gpu_bwd(p, o_bits, lse, deterministic=ORDERED)
    b = H.run_gpu_bwd(p, o_bits, lse, deterministic=ORDERED)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    _parity(p, deterministic=ORDERED)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_varlen_gqa_d64(dtype):
    """d = 64 with packed sequences and grouped-query heads (8 query heads on 2 kv heads), unequal
    query / key lengths per sequence, causal bottom-right."""
    lq = np.array([1, 200, 77, 129, 300]); lkv = np.array([5, 150, 260, 129, 310])
    p = synth.dense_problem("varlen_gqa64", dtype=dtype, b=len(lq), h=8, h_kv=2, d=64, lens_q=lq, lens_kv=lkv,
                            mask=BR, seed=22 + dtype)
    _parity(p)


@pytest.mark.parametrize("deterministic", [False, 2])
def test_workload1_full(deterministic):
    """fp16 b4 h12 s1024 d64 causal, BSHD viewed as BHSD: every output element (atomic and ordered dQ)."""
    _parity(synth.workload(1), deterministic=deterministic)


_ORACLE_CACHE = {}


def _oracle_full(idx):
    """Oracle forward (O rounded to 16 bits, LSE) and backward of workload idx, computed once per
    session: the atomic and deterministic tests of one workload share them."""
    if idx not in _ORACLE_CACHE:
        p = synth.workload(idx)
        o_bits, lse = H.oracle_forward(p)
        ref = oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                               p.f64("do"), lse, p.cu_q, p.cu_kv, p.scale, p.mask)
        _ORACLE_CACHE[idx] = (p, o_bits, lse, ref)
    return _ORACLE_CACHE[idx]


def _full_parity(idx, deterministic=False):
    """Every element of dQ, dK, dV against the oracle, plus the invariant
    sum_j dV_j = sum_i dO_i per (sequence, kv head group), which holds at any size."""
    p, o_bits, lse, (rq, rk, rv) = _oracle_full(idx)
    dq, dk, dv = H.run_gpu_bwd(p, o_bits, lse, deterministic)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")
    G = p.h // p.h_kv
    do = p.f64("do")
    for b in range(len(p.cu_kv)):
        s0, s1 = (0 if b == 0 else p.cu_kv[b - 1]), p.cu_kv[b]
        q0, q1 = (0 if b == 0 else p.cu_q[b - 1]), p.cu_q[b]
        for g in range(p.h_kv):
            want = do[q0:q1, g * G:(g + 1) * G].sum((0, 1))
            got = dv[s0:s1, g].sum(0)
            assert np.abs(got - want).max() <= 0.05 * np.abs(want).max() + 0.5
    return dq, dk, dv


@pytest.mark.slow
@pytest.mark.parametrize("deterministic", [False, True, ORDERED])
def test_workload2_full(deterministic):
    """bf16 b2 h32 s4096 d128 causal: every output element, all three dQ modes."""
    _full_parity(2, deterministic)


@pytest.mark.slow
@pytest.mark.parametrize("deterministic", [False, ORDERED])
def test_workload3_full(deterministic):
    """varlen GQA bf16, h 32 / h_kv 8, d128, 8 lengths in [256, 4096], causal bottom-right: every
    output element (atomic and ordered dQ)."""
    _full_parity(3, deterministic)


@pytest.mark.parametrize("idx", [1, 2])
def test_ordered_mode_workload_bitwise(idx):
    """Ordered dQ mode at the full workloads 1 and 2: two calls give the same bits."""
    if idx == 2:
        p, o_bits, lse, _ = _oracle_full(2)
    else:
        p = synth.workload(1)
        o_bits, lse = H.oracle_forward(p)
    a = H.run_gpu_bwd(p, o_bits, lse, ORDERED)
    b = H.run_gpu_bwd(p, o_bits, lse, ORDERED)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
