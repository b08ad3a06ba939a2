"""GPU parity of the NSA selected-attention forward (O, softmaxMax, softmaxSum),
of the backward with fp32 gradient outputs, and of the backward with a value
head dim unlike the query / key one (the Ascend page's Constraints: D is 192 or
128, K and V may differ; parameter table: FLOAT16 / BFLOAT16 / FLOAT32
outputs), all against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _problem(sparse_mode, dtype=synth.BF16, n1=16, n2=2, d=128, d_v=None, seed=1, lens_q=(300, 129),
             lens_kv=(512, 256), block_size=64, block_count=4):
    return synth.nsa_problem("nsa_ext", dtype=dtype, lens_q=list(lens_q), lens_kv=list(lens_kv), n1=n1, n2=n2,
                             d=d, d_v=d_v, block_size=block_size, block_count=block_count,
                             sparse_mode=sparse_mode, seed=seed)


def _fwd_parity(p):
    o, mx, sm, m8, s8 = H.run_gpu_nsa_fwd(p)
    ro, rmx, rsm = oracle.nsa_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.topk, p.cu_q, p.cu_kv, p.scale,
                                  p.block_size, p.sparse_mode)
    H.assert_close(o, ro, "O")
    fin = np.isfinite(rmx)
    assert np.all(np.isneginf(mx[~fin])) and np.all(sm[~fin] == 0), "rows without keys: max -inf, sum 0"
    np.testing.assert_allclose(mx[fin], rmx[fin], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(sm[fin], rsm[fin], rtol=1e-4)
    for lane in range(8):  # every lane of a stats row holds the same value
        np.testing.assert_array_equal(m8[..., lane], m8[..., 0])
        np.testing.assert_array_equal(s8[..., lane], s8[..., 0])


@pytest.mark.parametrize("sparse_mode", [0, 2])
@pytest.mark.parametrize("n1,n2", [(16, 2), (4, 1), (32, 1), (1, 1), (3, 1), (12, 1), (20, 2)])
def test_nsa_forward_parity(sparse_mode, n1, n2):
    """The tensor-core forward (two passes over the block lists: row maxima, then sums and O) for full
    and padded head groups, both sparse modes."""
    _fwd_parity(_problem(sparse_mode, n1=n1, n2=n2, seed=40 + n1 + sparse_mode))


@pytest.mark.parametrize("d,d_v", [(192, 128), (128, 192), (192, 192)])
def test_nsa_forward_unequal_dims(d, d_v):
    _fwd_parity(_problem(2, dtype=synth.F16, n1=8, n2=2, d=d, d_v=d_v, seed=50 + d + d_v, block_size=48,
                         lens_kv=(480, 240)))


def test_nsa_forward_workload4():
    """4 x 4096 tokens, 16 / 1 heads, d128, 16 blocks of 64, sparse mode 2: every element."""
    _fwd_parity(synth.workload(4))


def test_nsa_forward_bad_indices_flagged():
    import attention_backward_02_gb300 as ab
    p = _problem(0, seed=4)
    bad = p.topk.copy()
    bad[5, 0, 1] = 1000
    bad[7, 1, 2] = bad[7, 1, 0]
    H.run_gpu_nsa_fwd(p, topk=bad, expect_flags=ab._lib.ATTN_DEV_INDEX_RANGE | ab._lib.ATTN_DEV_INDEX_DUP)


def _bwd_parity(p, grad_fp32=False, deterministic=False):
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    dq, dk, dv = H.run_gpu_nsa(p, o_bits, mx, sm, deterministic=deterministic, grad_fp32=grad_fp32)
    rq, rk, rv = oracle.nsa_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                                p.f64("do"), mx.astype(np.float64), sm.astype(np.float64), p.topk, p.cu_q,
                                p.cu_kv, p.scale, p.block_size, p.sparse_mode)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")
    return dq, dk, dv


@pytest.mark.parametrize("n1,n2", [(16, 2), (4, 1)])
@pytest.mark.parametrize("deterministic", [False, True, 2])
def test_nsa_backward_fp32_gradients(n1, n2, deterministic):
    """fp32 dq / dk / dv on the tensor-core kernel: a full head group (16 / 2) and a padded one (4 / 1)."""
    p = _problem(2, n1=n1, n2=n2, seed=60 + n1)
    dq, dk, dv = _bwd_parity(p, grad_fp32=True, deterministic=deterministic)
    assert dq.dtype == np.float64  # fp32 values widened by the harness


@pytest.mark.parametrize("d,d_v", [(192, 128), (128, 192), (192, 192)])
@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_backward_unequal_dims(d, d_v, sparse_mode):
    p = _problem(sparse_mode, dtype=synth.BF16, n1=8, n2=2, d=d, d_v=d_v, seed=70 + d + d_v + sparse_mode,
                 block_size=48, lens_kv=(480, 240))
    _bwd_parity(p)


def test_nsa_backward_unequal_dims_fp32():
    p = _problem(2, dtype=synth.F16, n1=16, n2=1, d=192, d_v=128, seed=80)
    _bwd_parity(p, grad_fp32=True)


@pytest.mark.parametrize("mode", [True, 2])
def test_nsa_unequal_dims_deterministic_refused(mode):
    import attention_backward_02_gb300 as ab
    p = _problem(0, n1=16, n2=2, d=192, d_v=128, seed=81)
    o_bits, mx, sm = H.nsa_oracle_inputs(p)
    with pytest.raises(ab.AttnError) as e:
        H.run_gpu_nsa(p, o_bits, mx, sm, deterministic=mode)
    assert e.value.status == ab._lib.ATTN_ERR_UNSUPPORTED


# ------------------------------------------------ attenMaskOptional (2-D mask)

def _mask(rows, cols, seed, frac=0.3):
    return (np.random.default_rng(seed).random((rows, cols)) < frac).astype(np.uint8)


@pytest.mark.parametrize("sparse_mode", [0, 2])
@pytest.mark.parametrize("n1,n2", [(16, 2), (4, 1)])
def test_nsa_forward_with_mask(sparse_mode, n1, n2):
    p = _problem(sparse_mode, n1=n1, n2=n2, seed=90 + n1 + sparse_mode)
    mask = _mask(320, 512, 91 + sparse_mode)  # covers both sequences (and more)
    o, mx, sm, m8, s8 = H.run_gpu_nsa_fwd(p, mask=mask)
    ro, rmx, rsm = oracle.nsa_fwd(p.f64("q"), p.f64("k"), p.f64("v"), p.topk, p.cu_q, p.cu_kv, p.scale,
                                  p.block_size, p.sparse_mode, mask=mask)
    H.assert_close(o, ro, "O")
    fin = np.isfinite(rmx)
    assert np.all(np.isneginf(mx[~fin])) and np.all(sm[~fin] == 0)
    np.testing.assert_allclose(mx[fin], rmx[fin], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(sm[fin], rsm[fin], rtol=1e-4)


@pytest.mark.parametrize("sparse_mode", [0, 2])
@pytest.mark.parametrize("n1,n2,d,d_v,deterministic", [(16, 2, 128, 128, False), (4, 1, 128, 128, False),
                                                       (16, 2, 128, 128, True), (5, 1, 128, 128, True),
                                                       (16, 2, 128, 128, 2), (5, 1, 128, 128, 2),
                                                       (8, 2, 192, 128, False)])
def test_nsa_backward_with_mask(sparse_mode, n1, n2, d, d_v, deterministic):
    """The mask per element: on the tensor-core kernel (d = d_v = 128, both dQ modes, head groups of
    8, 4 and 5) and on the CUDA-core kernel (d = 192)."""
    p = _problem(sparse_mode, n1=n1, n2=n2, d=d, d_v=d_v, seed=92 + n1 + d + sparse_mode)
    mask = _mask(300, 512, 93 + n1 + sparse_mode)
    o_bits, mx, sm = H.nsa_oracle_inputs(p, mask=mask)
    dq, dk, dv = H.run_gpu_nsa(p, o_bits, mx, sm, mask=mask, deterministic=deterministic)
    rq, rk, rv = oracle.nsa_bwd(p.f64("q"), p.f64("k"), p.f64("v"), synth.bits_to_f64(o_bits, p.dtype),
                                p.f64("do"), mx.astype(np.float64), sm.astype(np.float64), p.topk, p.cu_q,
                                p.cu_kv, p.scale, p.block_size, p.sparse_mode, mask=mask)
    H.assert_close(dq, rq, "dQ")
    H.assert_close(dk, rk, "dK")
    H.assert_close(dv, rv, "dV")


def test_nsa_mask_too_small_refused():
    import attention_backward_02_gb300 as ab
    p = _problem(0, seed=94)
    with pytest.raises(ab.AttnError) as e:
        H.run_gpu_nsa_fwd(p, mask=_mask(300, 100, 95))  # narrower than the 512-key sequence
    assert e.value.status == ab._lib.ATTN_ERR_INVALID
