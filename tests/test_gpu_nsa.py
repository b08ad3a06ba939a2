"""GPU parity of the NSA selected-attention backward and its block lists
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _parity(p, deterministic=False):
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    dq, dk, dv = H.run_gpu_nsa(p, o_bits, mx, sm, deterministic)
    rq, rk, rv = oracle.nsa_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                                p.f64("do"), mx.astype(np.float64), sm.astype(np.float64), p.topk, p.cu_q,
                                p.cu_kv, p.scale, p.block_size, p.sparse_mode)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")
    return dq, dk, dv


def _small(sparse_mode, dtype=synth.BF16, seed=1, lens_q=(300, 129), lens_kv=(512, 256), n1=16, n2=2):
    return synth.nsa_problem("nsa_small", dtype=dtype, lens_q=list(lens_q), lens_kv=list(lens_kv), n1=n1, n2=n2,
                             d=128, block_size=64, block_count=4, sparse_mode=sparse_mode, seed=seed)


def _gpu_block_lists(p, topk=None):
    import torch
    import attention_backward_02_gb300 as ab
    starts = np.concatenate([[0], p.cu_kv[:-1]])
    nblk = int(((p.cu_kv - starts) // p.block_size).max())
    nrows = len(p.cu_q) * p.n2 * nblk
    offsets = torch.full((nrows + 1,), -1, dtype=torch.int32, device="cuda")
    tokens = torch.full((max(1, p.t1 * p.n2 * p.block_count),), -1, dtype=torch.int32, device="cuda")
    tk = torch.from_numpy(np.ascontiguousarray(p.topk if topk is None else topk, np.int32)).cuda()
    nblk_out, ws = ab.nsa_block_lists(H.nsa_desc(p), tk, offsets, tokens)
    flags = ab.attn_query_status(ws)
    off = offsets.cpu().numpy().astype(np.int64)
    return nblk_out, off, tokens.cpu().numpy()[: off[-1]], flags


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_block_lists_bit_exact(sparse_mode):
    p = _small(sparse_mode, seed=3)
    nblk, off, tok, flags = _gpu_block_lists(p)
    ref_off, ref_tok, ref_nblk = oracle.nsa_block_lists(p.topk, p.cu_q, p.cu_kv, p.n1, p.block_size, sparse_mode)
    assert flags == 0 and nblk == ref_nblk
    np.testing.assert_array_equal(off, ref_off)
    np.testing.assert_array_equal(tok, ref_tok)


def test_block_lists_workload4_bit_exact():
    p = synth.workload(4)
    nblk, off, tok, flags = _gpu_block_lists(p)
    ref_off, ref_tok, ref_nblk = oracle.nsa_block_lists(p.topk, p.cu_q, p.cu_kv, p.n1, p.block_size,
                                                        p.sparse_mode)
    assert flags == 0 and nblk == ref_nblk
    np.testing.assert_array_equal(off, ref_off)
    np.testing.assert_array_equal(tok, ref_tok)


def test_bad_indices_are_flagged_not_fatal():
    import attention_backward_02_gb300 as ab
    p = _small(0, seed=4)
    bad = p.topk.copy()
    bad[5, 0, 1] = 1000           # out of range
    bad[7, 1, 2] = bad[7, 1, 0]   # duplicate
    *_, flags = _gpu_block_lists(p, bad)
    assert flags == ab._lib.ATTN_DEV_INDEX_RANGE | ab._lib.ATTN_DEV_INDEX_DUP
    # the backward also completes, flags the same, and leaves a usable context
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    H.run_gpu_nsa(p, o_bits, mx, sm, topk=bad,
                  expect_flags=ab._lib.ATTN_DEV_INDEX_RANGE | ab._lib.ATTN_DEV_INDEX_DUP)
    _parity(p)  # a clean call afterwards is clean


@pytest.mark.parametrize("sparse_mode", [0, 2])
@pytest.mark.parametrize("dtype", [synth.F16, synth.BF16])
def test_small_parity(sparse_mode, dtype):
    _parity(_small(sparse_mode, dtype=dtype, seed=5 + sparse_mode))


def test_ascend_example_shape_is_dense():
    """selectedBlockCount * selectedBlockSize = S2 and topk = 0..cnt-1 selects
    every key: the GPU NSA result must match the oracle's dense backward."""
    p = synth.nsa_problem("dense_eq", dtype=synth.BF16, lens_q=[64], lens_kv=[1024], n1=16, n2=1, d=128,
                          block_size=64, block_count=16, sparse_mode=0, seed=6)
    p.topk[:] = np.arange(16, dtype=np.int32)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    dq, dk, dv = H.run_gpu_nsa(p, o_bits, mx, sm)
    lse = mx.astype(np.float64) + np.log(sm.astype(np.float64))
    rq, rk, rv = oracle.dense_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                                  p.f64("do"), lse, p.cu_q, p.cu_kv, p.scale, oracle.MASK_NONE)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")


def test_workload4_full():
    """NSA bf16, 4 x 4096 tokens, 16 query heads / 1 kv head, d128, 16 blocks of 64, sparse mode 2."""
    _parity(synth.workload(4))


@pytest.mark.parametrize("sparse_mode", [0, 2])
@pytest.mark.parametrize("n1,n2", [(16, 2), (16, 1), (32, 1)])
def test_deterministic_parity_and_bitwise(sparse_mode, n1, n2):
    """Deterministic mode: dQ from per-slot partials summed in slot order, one
    writer per dK / dV element; two calls give the same bits."""
    p = _small(sparse_mode, seed=11 + sparse_mode, n1=n1, n2=n2)
    first = _parity(p, deterministic=True)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    second = H.run_gpu_nsa(p, o_bits, mx, sm, deterministic=True)
    for a, b in zip(first, second):
        np.testing.assert_array_equal(a, b)


def test_deterministic_bad_indices_flagged():
    import attention_backward_02_gb300 as ab
    p = _small(2, seed=4)
    bad = p.topk.copy()
    bad[5, 0, 1] = 1000
    bad[7, 1, 2] = bad[7, 1, 0]
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    H.run_gpu_nsa(p, o_bits, mx, sm, deterministic=True, topk=bad,
                  expect_flags=ab._lib.ATTN_DEV_INDEX_RANGE | ab._lib.ATTN_DEV_INDEX_DUP)
    _parity(p, deterministic=True)


@pytest.mark.parametrize("n1,n2", [(8, 2), (3, 1), (12, 1), (20, 2)])
def test_deterministic_padded_groups(n1, n2):
    """Deterministic mode for head groups G = 4, 3, 12, 10 (rows padded to a multiple of 8 per token in
    the tensor-core kernel): oracle parity and the same bits from two calls."""
    p = _small(0, seed=12 + n1, n1=n1, n2=n2)
    first = _parity(p, deterministic=True)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    second = H.run_gpu_nsa(p, o_bits, mx, sm, deterministic=True)
    for x, y in zip(first, second):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("n1,n2", [(4, 1), (2, 2), (4, 2), (6, 3), (1, 1), (3, 1), (5, 1), (7, 1), (12, 1),
                                   (20, 1), (24, 1), (27, 1), (30, 3)])
@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_padded_head_groups(n1, n2, sparse_mode):
    """Head groups G = n1 / n2 that do not fill a 128-row chunk in whole tokens of G rows (1 to 30):
    each token's rows are padded to a multiple of 8 in the tensor-core kernel; both sparse modes."""
    _parity(_small(sparse_mode, seed=31 + n1 + n2 + sparse_mode, n1=n1, n2=n2))


def test_workload4_deterministic_bitwise():
    p = synth.workload(4)
    first = _parity(p, deterministic=True)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    second = H.run_gpu_nsa(p, o_bits, mx, sm, deterministic=True)
    for a, b in zip(first, second):
        np.testing.assert_array_equal(a, b)


# ------------------------------------------------ ordered deterministic mode (deterministic = 2)

def _two_runs_same_bits(p, mode):
    first = _parity(p, deterministic=mode)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    second = H.run_gpu_nsa(p, o_bits, mx, sm, mode)
    for a, b in zip(first, second):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("sparse_mode", [0, 2])
@pytest.mark.parametrize("n1,n2", [(16, 2), (16, 1), (32, 1)])
def test_ordered_parity_and_bitwise(sparse_mode, n1, n2):
    """One dQ accumulator whose adds for a token go in decreasing block order behind a counter per
    (token, kv head): oracle parity and the same bits from two calls."""
    _two_runs_same_bits(_small(sparse_mode, seed=41 + sparse_mode, n1=n1, n2=n2), 2)


@pytest.mark.parametrize("n1,n2", [(8, 2), (3, 1), (12, 1), (20, 2)])
def test_ordered_padded_groups(n1, n2):
    _two_runs_same_bits(_small(2, seed=52 + n1, n1=n1, n2=n2), 2)


def test_ordered_bad_indices_flagged():
    """An index out of range and a repeat are dropped by the block lists; the count of blocks a token waits
    for must drop them too, or the waits would run out."""
    import attention_backward_02_gb300 as ab
    p = _small(2, seed=4)
    bad = p.topk.copy()
    bad[5, 0, 1] = 1000
    bad[7, 1, 2] = bad[7, 1, 0]
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    H.run_gpu_nsa(p, o_bits, mx, sm, 2, topk=bad,
                  expect_flags=ab._lib.ATTN_DEV_INDEX_RANGE | ab._lib.ATTN_DEV_INDEX_DUP)


def test_workload4_ordered_bitwise():
    """4 x 4096 tokens, 16 / 1 heads, d128, 16 blocks of 64, sparse mode 2: every element, two calls."""
    _two_runs_same_bits(synth.workload(4), 2)
