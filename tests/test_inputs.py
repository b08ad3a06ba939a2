"""The seeded input recipe (CPU only): 16-bit rounding of the N(0,1) draws and
the NSA topk lists, checked against their stated definitions."""
import numpy as np
import pytest

import synth


def test_fp16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -2.5, 65504.0, 1e-8], np.float32)
    bits = synth.to_bits(x, synth.F16)
    np.testing.assert_array_equal(bits, x.astype(np.float16).view(np.uint16))
    # ties go to even: 1 + 2^-11 lies halfway between 1 and 1 + 2^-10
    assert synth.bits_to_f64(bits, synth.F16)[1] == 1.0
    assert synth.bits_to_f64(bits, synth.F16)[2] == 1.0 + 2.0 ** -9


def test_bf16_rounding_is_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4096).astype(np.float32),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -3.0e38, 0.0], np.float32)])
    ours = synth.to_bits(x, synth.BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(synth.bits_to_f64(ours, synth.BF16),
                                  torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def _check_topk(topk, cu_q, cu_kv, n2, bs, cnt, causal):
    starts_q = np.concatenate([[0], cu_q[:-1]]); starts_kv = np.concatenate([[0], cu_kv[:-1]])
    for b in range(len(cu_q)):
        lq, lkv = int(cu_q[b] - starts_q[b]), int(cu_kv[b] - starts_kv[b])
        nblk = lkv // bs
        for i in range(lq):
            for g in range(n2):
                ids = topk[starts_q[b] + i, g]
                assert len(set(ids.tolist())) == cnt, "distinct per (token, kv head)"
                assert ids.min() >= 0 and ids.max() < nblk, "local to the sequence, in range"
                if causal:
                    last = i + (lkv - lq)
                    nvis = min(nblk, last // bs + 1) if last >= 0 else 0
                    visible = set(range(nvis))
                    if nvis >= cnt:
                        assert set(ids.tolist()) <= visible
                        assert min(nblk - 1, last // bs) in set(ids.tolist()), "own block taken"
                    else:
                        assert visible <= set(ids.tolist()), "every visible block taken"
                        assert all(x >= nvis for x in set(ids.tolist()) - visible), "filler is fully masked"


@pytest.mark.parametrize("causal", [False, True])
def test_topk_follows_its_recipe(causal):
    rng = np.random.default_rng(3)
    cu_q, cu_kv = np.cumsum([300, 129, 64]), np.cumsum([512, 256, 1024])
    topk = synth.nsa_topk(rng, cu_q, cu_kv, 2, 64, 4, causal)
    assert topk.shape == (int(cu_q[-1]), 2, 4) and topk.dtype == np.int32
    _check_topk(topk, cu_q, cu_kv, 2, 64, 4, causal)


def test_nsa_workload_shapes_and_topk():
    """The NSA workload: 4 x 4096 tokens, 16 query heads / 1 kv head, d 128, 16 blocks of 64, sparse mode 2,
    scale 1/sqrt(128); its topk follows the causal recipe (checked on the first sequence)."""
    p = synth.workload(4)
    assert (p.t1, p.n1, p.n2, p.d, p.block_size, p.block_count, p.sparse_mode) == (16384, 16, 1, 128, 64, 16, 2)
    np.testing.assert_array_equal(np.diff(np.concatenate([[0], p.cu_q])), [4096] * 4)
    assert abs(p.scale - 128 ** -0.5) < 1e-12
    _check_topk(p.topk[:4096], p.cu_q[:1], p.cu_kv[:1], 1, 64, 16, True)


def test_dense_workload_shapes():
    """Workloads 0-3 as stated: sizes, dtype, scale, mask; workload 3's lengths are seeded draws from
    [256, 4096] (listed with the input recipe)."""
    w = {i: synth.workload(i) for i in range(4)}
    assert (w[0].dtype, w[0].b, w[0].h, w[0].h_kv, w[0].s_q, w[0].d, w[0].mask) == (synth.F16, 1, 2, 2, 128, 64, 0)
    assert (w[1].dtype, w[1].b, w[1].h, w[1].s_q, w[1].s_kv, w[1].d, w[1].mask) == (synth.F16, 4, 12, 1024, 1024, 64, 1)
    assert w[0].scale == w[1].scale == 0.125
    assert (w[2].dtype, w[2].b, w[2].h, w[2].s_q, w[2].d, w[2].mask) == (synth.BF16, 2, 32, 4096, 128, 1)
    assert abs(w[2].scale - 128 ** -0.5) < 1e-12
    lens = np.diff(np.concatenate([[0], w[3].cu_q])).tolist()
    assert lens == [3807, 2457, 3066, 2285, 2298, 3189, 2967, 3373]
    assert np.array_equal(w[3].cu_q, w[3].cu_kv) and (w[3].h, w[3].h_kv, w[3].d) == (32, 8, 128)
    assert w[3].varlen and w[3].mask == 2
