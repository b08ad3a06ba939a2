"""Seeded synthetic inputs for the attention-backward workloads.

This module only draws random numbers and rounds them to 16-bit storage; it
holds none of the attention arithmetic.  The tests, the smoke check and the
benchmark feed the same bits to the CUDA library and to the fp64 oracle.

Recipe (cuDNN-frontend SDPA-backward sample, cells "Problem sizes" and the
tensor set-up cell: N(0,1) draws cast to half precision, torch.manual_seed):
values are drawn in fp32 from numpy's PCG64 generator seeded with
``seed``, then rounded to fp16 or bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses

import numpy as np

F16, BF16 = 0, 1


def round_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x32, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_bits(x32: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp32 values to the 16-bit storage type; returns uint16 bit patterns."""
    if dtype == F16:
        return np.ascontiguousarray(x32, np.float32).astype(np.float16).view(np.uint16)
    return round_bf16_bits(x32)


def bits_to_f64(bits: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    return bf16_bits_to_f64(bits)


@dataclasses.dataclass
class DenseProblem:
    """A dense (optionally varlen / grouped-query) SDPA problem.

    Tensors are stored token-major: q, o, do are [Tq, h, d] and k, v are
    [Tkv, h_kv, d] uint16 bit patterns.  A fixed-length batch has
    cu_q = (s_q, 2 s_q, ...); its physical layout is then BSHD and the
    logical BHSD view has strides (s*h*d, d, h*d, 1).
    """
    name: str
    dtype: int
    b: int
    h: int
    h_kv: int
    d: int
    scale: float
    mask: int
    cu_q: np.ndarray
    cu_kv: np.ndarray
    varlen: bool
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray

    @property
    def s_q(self) -> int:
        return int(self.cu_q[0]) if not self.varlen else int(np.diff(np.concatenate([[0], self.cu_q])).max())

    @property
    def s_kv(self) -> int:
        return int(self.cu_kv[0]) if not self.varlen else int(np.diff(np.concatenate([[0], self.cu_kv])).max())

    @property
    def t_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def t_kv(self) -> int:
        return int(self.cu_kv[-1])

    def f64(self, name: str) -> np.ndarray:
        return bits_to_f64(getattr(self, name), self.dtype)


def _normal_bits(rng, shape, dtype):
    return to_bits(rng.standard_normal(shape, dtype=np.float32), dtype)


def dense_problem(name, *, dtype, b, h, h_kv, d, s_q=None, s_kv=None, lens_q=None, lens_kv=None,
                  scale=None, mask=0, seed=42) -> DenseProblem:
    """N(0,1) Q, K, V, dO rounded to 16 bits.  Fixed length when lens_* is None."""
    rng = np.random.default_rng(seed)
    varlen = lens_q is not None
    if varlen:
        lens_q = np.asarray(lens_q, np.int64)
        lens_kv = np.asarray(lens_kv if lens_kv is not None else lens_q, np.int64)
        b = len(lens_q)
    else:
        lens_q = np.full(b, s_q, np.int64)
        lens_kv = np.full(b, s_kv if s_kv is not None else s_q, np.int64)
    cu_q, cu_kv = np.cumsum(lens_q), np.cumsum(lens_kv)
    tq, tkv = int(cu_q[-1]), int(cu_kv[-1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q = _normal_bits(rng, (tq, h, d), dtype)
    k = _normal_bits(rng, (tkv, h_kv, d), dtype)
    v = _normal_bits(rng, (tkv, h_kv, d), dtype)
    do = _normal_bits(rng, (tq, h, d), dtype)
    return DenseProblem(name, dtype, b, h, h_kv, d, float(scale), mask, cu_q, cu_kv, varlen, q, k, v, do)


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n sequence lengths drawn uniformly from [lo, hi] (inclusive)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n).astype(np.int64)


@dataclasses.dataclass
class NsaProblem:
    """An NSA selected-attention problem in TND layout (uint16 bit patterns)."""
    name: str
    dtype: int
    n1: int
    n2: int
    d: int
    scale: float
    block_size: int
    block_count: int
    sparse_mode: int
    cu_q: np.ndarray
    cu_kv: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    topk: np.ndarray  # [T1, n2, cnt] int32

    @property
    def t1(self) -> int:
        return int(self.cu_q[-1])

    @property
    def t2(self) -> int:
        return int(self.cu_kv[-1])

    def f64(self, name: str) -> np.ndarray:
        return bits_to_f64(getattr(self, name), self.dtype)


def nsa_topk(rng, cu_q, cu_kv, n2, block_size, block_count, causal):
    """Block ids per (token, kv head), local to the token's sequence.

    causal: every block whose first key is visible to the token (its own
    block included) is taken first, in random order; if fewer than
    block_count exist, the rest are distinct blocks drawn from the later,
    fully masked ones.  Non-causal: block_count distinct blocks uniformly.
    """
    t1 = int(cu_q[-1])
    out = np.empty((t1, n2, block_count), np.int32)
    starts_q = np.concatenate([[0], cu_q[:-1]])
    starts_kv = np.concatenate([[0], cu_kv[:-1]])
    for bi in range(len(cu_q)):
        lq, lkv = int(cu_q[bi] - starts_q[bi]), int(cu_kv[bi] - starts_kv[bi])
        nblk = lkv // block_size
        for i in range(lq):
            t = int(starts_q[bi]) + i
            for g in range(n2):
                if causal:
                    last_visible_key = i + (lkv - lq)
                    nvis = min(nblk, last_visible_key // block_size + 1)
                    own = min(nblk - 1, max(0, last_visible_key) // block_size)
                    if nvis >= block_count:
                        others = np.delete(np.arange(nvis), own)
                        pick = rng.choice(others, block_count - 1, replace=False)
                        ids = np.concatenate([[own], pick])
                    else:
                        fill = rng.choice(np.arange(nvis, nblk), block_count - nvis, replace=False)
                        ids = np.concatenate([np.arange(nvis), fill])
                    rng.shuffle(ids)
                else:
                    ids = rng.choice(nblk, block_count, replace=False)
                out[t, g] = ids
    return out


def nsa_problem(name, *, dtype, lens_q, lens_kv=None, n1, n2, d, block_size, block_count,
                sparse_mode, scale=None, seed=42, d_v=None) -> NsaProblem:
    """d: query / key head dim; d_v: value head dim of v, O and dO (default d)."""
    rng = np.random.default_rng(seed)
    lens_q = np.asarray(lens_q, np.int64)
    lens_kv = np.asarray(lens_kv if lens_kv is not None else lens_q, np.int64)
    cu_q, cu_kv = np.cumsum(lens_q), np.cumsum(lens_kv)
    t1, t2 = int(cu_q[-1]), int(cu_kv[-1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q = _normal_bits(rng, (t1, n1, d), dtype)
    k = _normal_bits(rng, (t2, n2, d), dtype)
    v = _normal_bits(rng, (t2, n2, d if d_v is None else d_v), dtype)
    do = _normal_bits(rng, (t1, n1, d if d_v is None else d_v), dtype)
    topk = nsa_topk(rng, cu_q, cu_kv, n2, block_size, block_count, causal=(sparse_mode == 2))
    return NsaProblem(name, dtype, n1, n2, d, float(scale), block_size, block_count, sparse_mode,
                      cu_q, cu_kv, q, k, v, do, topk)


# --------------------------------------------------------------------------
# the five workloads (seed 42 + index)
# --------------------------------------------------------------------------

def workload(idx: int, seed=None, **over):
    """Workload idx in 0..4, with the sizes of the pages' problems:

    0  dense fwd+bwd, fp16, b1 h2 s128 d64, scale 1/8, non-causal
    1  dense bwd, fp16, b4 h12 s1024 d64, scale 1/8, causal (GPT-2 sizes)
    2  dense bwd, bf16, b2 h32 s4096 d128, causal
    3  varlen GQA, bf16, 8 sequences with lengths U[256,4096], h 32 / h_kv 8,
       d128, causal bottom-right
    4  NSA selected attention, bf16, 4 x 4096 tokens, n1 16 / n2 1, d128,
       block 64 x 16, sparse mode 2
    """
    seed = 42 + idx if seed is None else int(seed)  # another seed: another shard of the same shape
    if idx == 0:
        kw = dict(dtype=F16, b=1, h=2, h_kv=2, d=64, s_q=128, s_kv=128, scale=1 / 8, mask=0)
    elif idx == 1:
        kw = dict(dtype=F16, b=4, h=12, h_kv=12, d=64, s_q=1024, s_kv=1024, scale=1 / 8, mask=1)
    elif idx == 2:
        kw = dict(dtype=BF16, b=2, h=32, h_kv=32, d=128, s_q=4096, s_kv=4096, scale=1 / np.sqrt(128), mask=1)
    elif idx == 3:
        lens = varlen_lengths(8, 256, 4096, seed)
        kw = dict(dtype=BF16, b=8, h=32, h_kv=8, d=128, lens_q=lens, lens_kv=lens,
                  scale=1 / np.sqrt(128), mask=2)
    elif idx == 4:
        kw = dict(dtype=BF16, lens_q=[4096] * 4, n1=16, n2=1, d=128, block_size=64, block_count=16,
                  sparse_mode=2, scale=1 / np.sqrt(128))
        kw.update(over)
        return nsa_problem(f"nsa{idx}", seed=seed, **kw)
    else:
        raise ValueError(idx)
    kw.update(over)
    return dense_problem(f"dense{idx}", seed=seed, **kw)
