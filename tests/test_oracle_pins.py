"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test pins the oracle to something it cannot agree with by construction:
hand-worked closed forms (tests/golden), finite differences of the forward,
exact invariants of the softmax gradient, special cases that reduce to plain
averages, the Ascend NSA example (which is dense attention in disguise), an
independent masked-dense NSA path, and PyTorch fp64 autograd of the
matmul -> scale -> softmax -> matmul pattern.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import CAUSAL_BOTTOM_RIGHT, CAUSAL_TOP_LEFT, MASK_NONE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- closed forms

def test_two_keys_closed_form():
    g = _golden("two_keys.json")
    q = np.array(g["q"])[:, None, :]
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    do = np.array(g["do"])[:, None, :]
    o, lse = oracle.dense_fwd(q, k, v, [1], [2], g["scale"])
    np.testing.assert_allclose(o[:, 0], g["o"], rtol=1e-14)
    np.testing.assert_allclose(lse[:, 0], g["lse"], rtol=1e-14)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, [1], [2], g["scale"])
    np.testing.assert_allclose(dq[:, 0], g["dq"], rtol=1e-14)
    np.testing.assert_allclose(dk[:, 0], g["dk"], rtol=1e-14)
    np.testing.assert_allclose(dv[:, 0], g["dv"], rtol=1e-14)


@pytest.mark.parametrize("mask,key", [(MASK_NONE, "none"), (CAUSAL_TOP_LEFT, "top_left"),
                                      (CAUSAL_BOTTOM_RIGHT, "bottom_right")])
def test_mask_bitmaps(mask, key):
    """scale = 0 and one-hot value rows make O_i the indicator of the visible
    keys divided by their count, so the mask can be read off O."""
    g = _golden("causal_masks.json")
    sq, skv = g["s_q"], g["s_kv"]
    q = _rng(1).standard_normal((sq, 1, skv))
    k = _rng(2).standard_normal((skv, 1, skv))
    v = np.eye(skv)[:, None, :]
    o, _ = oracle.dense_fwd(q, k, v, [sq], [skv], 0.0, mask)
    bitmap = (o[:, 0, :] > 0).astype(int)
    assert bitmap.tolist() == g[key]
    np.testing.assert_allclose(o[:, 0, :].sum(-1), 1.0, rtol=1e-15)


# ------------------------------------------------------------ finite differences

def _loss_dense(q, k, v, do, cu_q, cu_kv, scale, mask):
    o, _ = oracle.dense_fwd(q, k, v, cu_q, cu_kv, scale, mask, threads=1)
    return float((o * do).sum())


def _fd_grad(f, x, eps=1e-5):
    g = np.zeros_like(x)
    flat, gflat = x.reshape(-1), g.reshape(-1)
    for idx in range(flat.size):
        old = flat[idx]
        flat[idx] = old + eps
        lp = f()
        flat[idx] = old - eps
        lm = f()
        flat[idx] = old
        gflat[idx] = (lp - lm) / (2 * eps)
    return g


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _check_dense_fd(lens_q, lens_kv, h, h_kv, d, scale, mask, seed):
    rng = _rng(seed)
    cu_q, cu_kv = np.cumsum(lens_q), np.cumsum(lens_kv)
    q = rng.standard_normal((cu_q[-1], h, d))
    k = rng.standard_normal((cu_kv[-1], h_kv, d))
    v = rng.standard_normal((cu_kv[-1], h_kv, d))
    do = rng.standard_normal((cu_q[-1], h, d))
    o, lse = oracle.dense_fwd(q, k, v, cu_q, cu_kv, scale, mask, threads=1)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, cu_q, cu_kv, scale, mask, threads=1)
    f = lambda: _loss_dense(q, k, v, do, cu_q, cu_kv, scale, mask)
    # rows without a visible key have no gradient and no O; fd gives 0 there too
    for name, x, g in (("dq", q, dq), ("dk", k, dk), ("dv", v, dv)):
        fd = _fd_grad(f, x)
        assert np.abs(fd - g).max() <= 1e-7 * max(1.0, np.abs(fd).max()), name


@pytest.mark.parametrize("mask", [MASK_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT])
@pytest.mark.parametrize("s_q", [1, 3, 7])
@pytest.mark.parametrize("s_kv", [1, 5, 9])
def test_dense_finite_differences(mask, s_q, s_kv):
    _check_dense_fd([s_q], [s_kv], h=2, h_kv=1, d=4, scale=0.7, mask=mask, seed=s_q * 31 + s_kv)


@pytest.mark.parametrize("mask", [MASK_NONE, CAUSAL_BOTTOM_RIGHT])
def test_dense_finite_differences_varlen_gqa(mask):
    _check_dense_fd([3, 6], [5, 6], h=4, h_kv=2, d=3, scale=0.9, mask=mask, seed=7)


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("mask", [MASK_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT])
def test_softmax_gradient_invariants(mask):
    """With exact O: sum_j dS_ij = 0 for every row, so sum_j dK_j = 0 per
    (sequence, kv head); and sum_j P_ij = 1, so sum_j dV_j = sum_i dO_i
    over the group's query rows that see at least one key."""
    rng = _rng(11)
    lens = np.array([5, 12, 9])
    cu = np.cumsum(lens)
    h, h_kv, d = 6, 2, 8
    q = rng.standard_normal((cu[-1], h, d))
    k = rng.standard_normal((cu[-1], h_kv, d))
    v = rng.standard_normal((cu[-1], h_kv, d))
    do = rng.standard_normal((cu[-1], h, d))
    o, lse = oracle.dense_fwd(q, k, v, cu, cu, 0.5, mask)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, cu, cu, 0.5, mask)
    starts = np.concatenate([[0], cu[:-1]])
    for b in range(len(lens)):
        sl = slice(starts[b], cu[b])
        for g in range(h_kv):
            np.testing.assert_allclose(dk[sl, g].sum(0), 0.0, atol=1e-12)
            heads = slice(g * (h // h_kv), (g + 1) * (h // h_kv))
            np.testing.assert_allclose(dv[sl, g].sum(0), do[sl, heads].sum((0, 1)), rtol=1e-12)
    # O is a convex combination of the value rows: all-ones values give O = 1
    o1, _ = oracle.dense_fwd(q, k, np.ones_like(v), cu, cu, 0.5, mask)
    np.testing.assert_allclose(o1, 1.0, rtol=1e-14)


def test_formula_mode_uses_supplied_o():
    """dS_ij = P_ij (dP_ij - D_i) with D from the supplied O: shifting O by a
    vector orthogonal to dO leaves every gradient unchanged; shifting along
    dO changes D_i by |dO_i|^2 and dQ by -scale |dO_i|^2 sum_j P_ij k_j."""
    rng = _rng(5)
    q = rng.standard_normal((4, 1, 3)); k = rng.standard_normal((6, 1, 3))
    v = rng.standard_normal((6, 1, 3)); do = rng.standard_normal((4, 1, 3))
    o, lse = oracle.dense_fwd(q, k, v, [4], [6], 0.8)
    base = oracle.dense_bwd(q, k, v, o, do, lse, [4], [6], 0.8)
    w = rng.standard_normal((4, 1, 3))
    w -= (w * do).sum(-1, keepdims=True) / (do * do).sum(-1, keepdims=True) * do
    same = oracle.dense_bwd(q, k, v, o + w, do, lse, [4], [6], 0.8)
    for a, b in zip(base, same):
        np.testing.assert_allclose(a, b, atol=1e-13)
    shifted = oracle.dense_bwd(q, k, v, o + do, do, lse, [4], [6], 0.8)
    p = np.exp(0.8 * q[:, 0] @ k[:, 0].T - lse)  # P of the definition
    expect_dq = base[0][:, 0] - 0.8 * (do[:, 0] ** 2).sum(-1, keepdims=True) * (p @ k[:, 0])
    np.testing.assert_allclose(shifted[0][:, 0], expect_dq, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- special cases

def test_single_key():
    """s_kv = 1: P = 1, so dQ = dK = 0 and dV = sum of dO over rows and heads."""
    rng = _rng(3)
    q = rng.standard_normal((5, 4, 8)); k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8)); do = rng.standard_normal((5, 4, 8))
    o, lse = oracle.dense_fwd(q, k, v, [5], [1], 0.3)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, [5], [1], 0.3)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0], do[:, 0:2].sum((0, 1)), rtol=1e-13)
    np.testing.assert_allclose(dv[0, 1], do[:, 2:4].sum((0, 1)), rtol=1e-13)


def test_constant_values_zero_ds():
    """Equal value rows: O_i = v, dP_ij = D_i, dS = 0, so dQ = dK = 0."""
    rng = _rng(4)
    q = rng.standard_normal((7, 2, 5)); k = rng.standard_normal((9, 2, 5))
    v = np.tile(rng.standard_normal((1, 2, 5)), (9, 1, 1)); do = rng.standard_normal((7, 2, 5))
    o, lse = oracle.dense_fwd(q, k, v, [7], [9], 0.6, CAUSAL_BOTTOM_RIGHT)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, [7], [9], 0.6, CAUSAL_BOTTOM_RIGHT)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)


def test_zero_scale_uniform_p():
    """scale = 0: P is uniform over the visible keys, so O_i is their mean and
    dV_j = sum over the rows that see j of dO_i / n_visible(i)."""
    rng = _rng(6)
    sq = skv = 6
    q = rng.standard_normal((sq, 1, 3)); k = rng.standard_normal((skv, 1, 3))
    v = rng.standard_normal((skv, 1, 3)); do = rng.standard_normal((sq, 1, 3))
    o, lse = oracle.dense_fwd(q, k, v, [sq], [skv], 0.0, CAUSAL_TOP_LEFT)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, [sq], [skv], 0.0, CAUSAL_TOP_LEFT)
    for i in range(sq):
        np.testing.assert_allclose(o[i, 0], v[: i + 1, 0].mean(0), rtol=1e-13)
    for j in range(skv):
        expect = sum(do[i, 0] / (i + 1) for i in range(j, sq))
        np.testing.assert_allclose(dv[j, 0], expect, rtol=1e-13)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)  # scale multiplies dQ and dK
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)


def test_empty_rows_bottom_right():
    """s_q > s_kv, bottom-right: the first s_q - s_kv rows see no key and get
    O = 0, LSE = +inf and zero gradient."""
    rng = _rng(8)
    q = rng.standard_normal((6, 1, 4)); k = rng.standard_normal((3, 1, 4))
    v = rng.standard_normal((3, 1, 4)); do = rng.standard_normal((6, 1, 4))
    o, lse = oracle.dense_fwd(q, k, v, [6], [3], 0.5, CAUSAL_BOTTOM_RIGHT)
    assert np.all(np.isinf(lse[:3])) and np.all(np.isfinite(lse[3:]))
    np.testing.assert_array_equal(o[:3], 0.0)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, [6], [3], 0.5, CAUSAL_BOTTOM_RIGHT)
    np.testing.assert_array_equal(dq[:3], 0.0)
    _check_dense_fd([6], [3], 1, 1, 4, 0.5, CAUSAL_BOTTOM_RIGHT, seed=8)


def test_sampled_rows_equal_full():
    rng = _rng(9)
    lens = np.array([7, 13]); cu = np.cumsum(lens)
    h, h_kv, d = 4, 2, 6
    q = rng.standard_normal((cu[-1], h, d)); k = rng.standard_normal((cu[-1], h_kv, d))
    v = rng.standard_normal((cu[-1], h_kv, d)); do = rng.standard_normal((cu[-1], h, d))
    o, lse = oracle.dense_fwd(q, k, v, cu, cu, 0.4, CAUSAL_TOP_LEFT)
    o = o + 0.01 * rng.standard_normal(o.shape)  # formula mode: O as supplied
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, cu, cu, 0.4, CAUSAL_TOP_LEFT)
    # rows of both sequences, including the last token of the first (6) and the first of the second (7)
    qr = np.array([0, 5, 17, 27, 29, 40, 79]); kr = np.array([0, 3, 12, 15, 20, 39])
    sdq, sdk, sdv = oracle.dense_bwd_rows(q, k, v, o, do, lse, cu, cu, 0.4, CAUSAL_TOP_LEFT, qr, kr)
    np.testing.assert_allclose(sdq, dq.reshape(-1, d)[qr], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sdk, dk.reshape(-1, d)[kr], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sdv, dv.reshape(-1, d)[kr], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------- PyTorch autograd

@pytest.mark.parametrize("mask", [MASK_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT])
def test_torch_autograd_crosscheck(mask):
    """PyTorch fp64 autograd of matmul -> scale -> (mask) -> softmax -> matmul,
    the pattern the PyTorch PR #94729 rewrites into an sdpa call (with the
    scale multiplied, not divided)."""
    torch = pytest.importorskip("torch")
    rng = _rng(12)
    sq, skv, d, scale = 5, 8, 4, 0.45
    q = rng.standard_normal((sq, 1, d)); k = rng.standard_normal((skv, 1, d))
    v = rng.standard_normal((skv, 1, d)); do = rng.standard_normal((sq, 1, d))
    o, lse = oracle.dense_fwd(q, k, v, [sq], [skv], scale, mask)
    dq, dk, dv = oracle.dense_bwd(q, k, v, o, do, lse, [sq], [skv], scale, mask)
    tq, tk, tv = (torch.tensor(x[:, 0], requires_grad=True) for x in (q, k, v))
    s = torch.matmul(tq, tk.transpose(-2, -1)) * scale
    i = torch.arange(sq)[:, None]; j = torch.arange(skv)[None, :]
    if mask == CAUSAL_TOP_LEFT:
        s = s.masked_fill(j > i, float("-inf"))
    elif mask == CAUSAL_BOTTOM_RIGHT:
        s = s.masked_fill(j > i + (skv - sq), float("-inf"))
    to = torch.matmul(torch.softmax(s, -1), tv)
    to.backward(torch.tensor(do[:, 0]))
    np.testing.assert_allclose(o[:, 0], to.detach().numpy(), rtol=1e-12)
    np.testing.assert_allclose(dq[:, 0], tq.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dk[:, 0], tk.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dv[:, 0], tv.grad.numpy(), rtol=1e-11, atol=1e-14)


# ------------------------------------------------------------------------- NSA

def _nsa_random(lens_q, lens_kv, n1, n2, d, bs, cnt, sparse_mode, seed):
    import synth
    rng = _rng(seed)
    cu_q, cu_kv = np.cumsum(lens_q), np.cumsum(lens_kv)
    q = rng.standard_normal((cu_q[-1], n1, d)); k = rng.standard_normal((cu_kv[-1], n2, d))
    v = rng.standard_normal((cu_kv[-1], n2, d)); do = rng.standard_normal((cu_q[-1], n1, d))
    topk = synth.nsa_topk(rng, cu_q, cu_kv, n2, bs, cnt, causal=(sparse_mode == 2))
    return cu_q, cu_kv, q, k, v, do, topk


def test_ascend_example_closed_form():
    g = _golden("ascend_nsa_example.json")
    t1, t2, d = g["s1"], g["s2"], g["d"]
    fill = g["fill"]
    q = np.full((t1, 1, d), fill); k = np.full((t2, 1, d), fill); v = np.full((t2, 1, d), fill)
    do = np.full((t1, 1, d), fill); o = np.full((t1, 1, d), fill)
    topk = np.array(g["topk"], np.int32).reshape(t1, 1, g["block_count"])
    o_f, mx, sm = oracle.nsa_fwd(q, k, v, topk, g["cu_q"], g["cu_kv"], g["scale"], g["block_size"],
                                 g["sparse_mode"])
    np.testing.assert_allclose(o_f, o, rtol=1e-15)
    np.testing.assert_allclose(mx, g["softmax_max"], rtol=1e-15)
    np.testing.assert_allclose(sm, g["softmax_sum"], rtol=1e-15)
    dq, dk, dv = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, g["cu_q"], g["cu_kv"], g["scale"],
                                g["block_size"], g["sparse_mode"])
    np.testing.assert_allclose(dq, g["dq"], atol=1e-12)
    np.testing.assert_allclose(dk, g["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, g["dv"], rtol=1e-13)


@pytest.mark.parametrize("sparse_mode,mask", [(0, MASK_NONE), (2, CAUSAL_BOTTOM_RIGHT)])
def test_ascend_example_shape_equals_dense(sparse_mode, mask):
    """With selectedBlockCount * selectedBlockSize = S2 and topk = 0..cnt-1 the
    selection is every key, so NSA is dense attention (the Ascend example's
    shape, random inputs); sparse mode 2 is then causal bottom-right."""
    rng = _rng(13)
    s1, s2, d, bs, cnt = 3, 1024, 192, 64, 16
    q = rng.standard_normal((s1, 1, d)) * 0.2; k = rng.standard_normal((s2, 1, d)) * 0.2
    v = rng.standard_normal((s2, 1, d)); do = rng.standard_normal((s1, 1, d))
    topk = np.tile(np.arange(cnt, dtype=np.int32), (s1, 1, 1))
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, [s1], [s2], 1.0, bs, sparse_mode)
    od, lse = oracle.dense_fwd(q, k, v, [s1], [s2], 1.0, mask)
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(mx + np.log(sm), lse, rtol=1e-13)
    got = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, [s1], [s2], 1.0, bs, sparse_mode)
    ref = oracle.dense_bwd(q, k, v, od, do, lse, [s1], [s2], 1.0, mask)
    for a, b in zip(got, ref):
        assert _rel(a, b) < 1e-12


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_finite_differences(sparse_mode):
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([8, 6], [8, 6], 4, 2, 3, 2, 2, sparse_mode, seed=21)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1)
    dq, dk, dv = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1)

    def loss():
        oo, _, _ = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1)
        return float((oo * do).sum())

    for name, x, g in (("dq", q, dq), ("dk", k, dk), ("dv", v, dv)):
        fd = _fd_grad(loss, x)
        assert np.abs(fd - g).max() <= 1e-7 * max(1.0, np.abs(fd).max()), name


def _nsa_random_dims(lens_q, lens_kv, n1, n2, d, d_v, bs, cnt, sparse_mode, seed):
    """As _nsa_random, with value / O / dO head dim d_v != d (the Ascend page allows 192 / 128)."""
    cu_q, cu_kv, q, k, _, _, topk = _nsa_random(lens_q, lens_kv, n1, n2, d, bs, cnt, sparse_mode, seed)
    rng = _rng(seed + 1000)
    v = rng.standard_normal((cu_kv[-1], n2, d_v)); do = rng.standard_normal((cu_q[-1], n1, d_v))
    return cu_q, cu_kv, q, k, v, do, topk


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_finite_differences_unequal_dims(sparse_mode):
    """Query / key head dim 2, value head dim 3: every gradient against central differences."""
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random_dims([8, 6], [8, 6], 4, 2, 2, 3, 2, 2, sparse_mode, seed=25)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1)
    assert o.shape == (cu_q[-1], 4, 3)
    dq, dk, dv = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape

    def loss():
        oo, _, _ = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1)
        return float((oo * do).sum())

    for name, x, g in (("dq", q, dq), ("dk", k, dk), ("dv", v, dv)):
        fd = _fd_grad(loss, x)
        assert np.abs(fd - g).max() <= 1e-7 * max(1.0, np.abs(fd).max()), name


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_gather_equals_masked_dense_unequal_dims(sparse_mode):
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random_dims([64, 40], [64, 48], 8, 2, 24, 16, 8, 3, sparse_mode,
                                                        seed=26)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, sparse_mode)
    got = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.3, 8, sparse_mode)
    od, *ref = oracle.nsa_masked_dense(q, k, v, do, topk, cu_q, cu_kv, 0.3, 8, sparse_mode)
    assert _rel(o, od) < 1e-12
    for a, b in zip(got, ref):
        assert _rel(a, b) < 1e-12


def test_nsa_rejects_mismatched_head_dims():
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random_dims([8], [8], 2, 1, 4, 3, 2, 2, 0, seed=27)
    with pytest.raises(ValueError):
        oracle.nsa_fwd(q, k[..., :3], v, topk, cu_q, cu_kv, 0.8, 2, 0)  # key head dim != query head dim
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, 0)
    with pytest.raises(ValueError):
        oracle.nsa_bwd(q, k, v, o, do[..., :2], mx, sm, topk, cu_q, cu_kv, 0.8, 2, 0)  # dY not value-dim


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_gather_equals_masked_dense(sparse_mode):
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([64, 40], [64, 48], 8, 2, 16, 8, 3, sparse_mode, seed=22)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, sparse_mode)
    got = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.3, 8, sparse_mode)
    od, *ref = oracle.nsa_masked_dense(q, k, v, do, topk, cu_q, cu_kv, 0.3, 8, sparse_mode)
    assert _rel(o, od) < 1e-12
    for a, b in zip(got, ref):
        assert _rel(a, b) < 1e-12


def test_nsa_rejects_out_of_range_index():
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([8], [8], 2, 1, 3, 2, 2, 0, seed=23)
    topk = topk.copy(); topk[3, 0, 1] = 4  # blocks of 2 keys: valid ids are 0..3
    with pytest.raises(ValueError):
        oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, 0)


def check_nsa_rejects_repeated_index():
    """A block id repeated within one (token, kv head) would count its keys
    twice under the gather: every NSA entry point refuses it."""
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([8], [8], 2, 1, 3, 2, 2, 0, seed=23)
    topk = topk.copy(); topk[3, 0, 1] = topk[3, 0, 0]
    o, mx, sm = np.zeros_like(q), np.ones(q.shape[:2]), np.ones(q.shape[:2])
    calls = {
        "nsa_fwd": lambda: oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, 0),
        "nsa_bwd": lambda: oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.8, 2, 0),
        "nsa_masked_dense": lambda: oracle.nsa_masked_dense(q, k, v, do, topk, cu_q, cu_kv, 0.8, 2, 0),
    }
    for name, call in calls.items():
        try:
            call()
        except ValueError:
            continue
        raise AssertionError(f"{name} accepted a repeated block id")


def test_nsa_rejects_repeated_index():
    check_nsa_rejects_repeated_index()


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_block_lists_definition(sparse_mode):
    """Block lists against a set-based construction with numpy."""
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([40, 24], [48, 24], 4, 2, 4, 8, 3, sparse_mode, seed=24)
    offsets, tokens, nblk = oracle.nsa_block_lists(topk, cu_q, cu_kv, 4, 8, sparse_mode)
    starts_q = np.concatenate([[0], cu_q[:-1]]); starts_kv = np.concatenate([[0], cu_kv[:-1]])
    pos = 0
    for b in range(len(cu_q)):
        lq, lkv = cu_q[b] - starts_q[b], cu_kv[b] - starts_kv[b]
        for g in range(2):
            for blk in range(nblk):
                toks = np.where((topk[starts_q[b]:cu_q[b], g, :] == blk).any(-1))[0]
                if sparse_mode == 2:
                    toks = toks[blk * 8 <= toks + (lkv - lq)]
                got = tokens[offsets[(b * 2 + g) * nblk + blk]: offsets[(b * 2 + g) * nblk + blk + 1]]
                np.testing.assert_array_equal(got, toks + starts_q[b])
                pos += len(toks)
    assert offsets[-1] == pos


# ------------------------------------------------ attenMaskOptional (2-D mask)
# Reading of the Ascend page's attenMaskOptional (2-D BOOL / UINT8, in the signature and the parameter
# table, used by no formula): entry (i, j) nonzero removes key j for query i, positions local to the
# sequence, on top of the selection and the sparse mode.

def test_nsa_zero_mask_is_no_mask():
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([64, 40], [64, 48], 8, 2, 16, 8, 3, 2, seed=31)
    zero = np.zeros((64, 64), np.uint8)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, 2)
    om, mxm, smm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, 2, mask=zero)
    np.testing.assert_array_equal(o, om)
    np.testing.assert_array_equal(mx, mxm)
    np.testing.assert_array_equal(sm, smm)
    a = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.3, 8, 2)
    b = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.3, 8, 2, mask=zero)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_nsa_causal_mask_equals_sparse_mode_2():
    """sparseMode 0 with the bottom-right causal pattern as attenMaskOptional is sparseMode 2."""
    lq, lkv = 24, 40
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([lq, lq], [lkv, lkv], 8, 2, 16, 8, 3, 2, seed=32)
    i, j = np.meshgrid(np.arange(lq), np.arange(lkv), indexing="ij")
    causal = (j > i + (lkv - lq)).astype(np.uint8)
    o2, mx2, sm2 = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, 2)
    o0, mx0, sm0 = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, 0, mask=causal)
    assert _rel(o0, o2) < 1e-14 and _rel(sm0, sm2) < 1e-14
    np.testing.assert_array_equal(mx0, mx2)
    a = oracle.nsa_bwd(q, k, v, o2, do, mx2, sm2, topk, cu_q, cu_kv, 0.3, 8, 2)
    b = oracle.nsa_bwd(q, k, v, o2, do, mx2, sm2, topk, cu_q, cu_kv, 0.3, 8, 0, mask=causal)
    for x, y in zip(a, b):
        assert _rel(y, x) < 1e-14


def test_nsa_mask_keeps_one_key_closed_form():
    """A mask that leaves each query exactly one key of its selection: P = 1 on that key, so O is
    that key's value row, softmaxSum = 1, softmaxMax = its score (the mask removes, it does not keep)."""
    rng = _rng(33)
    lq, lkv, d = 6, 8, 4
    q = rng.standard_normal((lq, 1, d)); k = rng.standard_normal((lkv, 1, d)); v = rng.standard_normal((lkv, 1, d))
    topk = np.tile(np.array([0, 1], np.int32), (lq, 1, 1))  # blocks of 4: every key selected
    keep = np.array([3, 0, 7, 5, 1, 6])
    mask = np.ones((lq, lkv), np.uint8)
    mask[np.arange(lq), keep] = 0
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, [lq], [lkv], 0.5, 4, 0, mask=mask)
    np.testing.assert_allclose(o[:, 0], v[keep, 0], rtol=1e-15)
    np.testing.assert_allclose(sm[:, 0], 1.0, rtol=1e-15)
    np.testing.assert_allclose(mx[:, 0], 0.5 * np.einsum("id,id->i", q[:, 0], k[keep, 0]), rtol=1e-14)


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_mask_finite_differences(sparse_mode):
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([8, 6], [8, 6], 4, 2, 3, 2, 2, sparse_mode, seed=34)
    mask = (_rng(35).random((8, 8)) < 0.3).astype(np.uint8)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1, mask=mask)
    dq, dk, dv = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1,
                                mask=mask)

    def loss():
        oo, _, _ = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, sparse_mode, threads=1, mask=mask)
        return float((oo * do).sum())

    for name, x, g in (("dq", q, dq), ("dk", k, dk), ("dv", v, dv)):
        fd = _fd_grad(loss, x)
        assert np.abs(fd - g).max() <= 1e-7 * max(1.0, np.abs(fd).max()), name


@pytest.mark.parametrize("sparse_mode", [0, 2])
def test_nsa_mask_gather_equals_masked_dense(sparse_mode):
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([64, 40], [64, 48], 8, 2, 16, 8, 3, sparse_mode, seed=36)
    mask = (_rng(37).random((64, 64)) < 0.25).astype(np.uint8)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.3, 8, sparse_mode, mask=mask)
    got = oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, cu_kv, 0.3, 8, sparse_mode, mask=mask)
    od, *ref = oracle.nsa_masked_dense(q, k, v, do, topk, cu_q, cu_kv, 0.3, 8, sparse_mode, mask=mask)
    assert _rel(o, od) < 1e-12
    for a, b in zip(got, ref):
        assert _rel(a, b) < 1e-12


def test_nsa_mask_must_cover_the_sequences():
    cu_q, cu_kv, q, k, v, do, topk = _nsa_random([8], [8], 2, 1, 3, 2, 2, 0, seed=38)
    with pytest.raises(ValueError):
        oracle.nsa_fwd(q, k, v, topk, cu_q, cu_kv, 0.8, 2, 0, mask=np.zeros((8, 7), np.uint8))
