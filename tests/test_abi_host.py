"""Host-only checks of the C ABI: the library loads, exports every declared
symbol, sizes workspaces, and rejects bad arguments before any launch.
No call here reaches a kernel, so none needs a GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ab():
    from attention_backward_02_gb300 import build
    build.build()
    import attention_backward_02_gb300 as ab
    ab._lib.load()
    return ab


def _declared():
    text = open(os.path.join(ROOT, "include", "attnbwd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))


def test_exports_every_declared_symbol(ab):
    names = _declared()
    assert names == set(ab._lib.EXPORTS), names
    lib = C.CDLL(ab._lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def _desc(ab, **kw):
    base = dict(dtype=ab.ATTN_F16, b=4, h=12, h_kv=12, s_q=1024, s_kv=1024, d=64, scale=0.125,
                mask=ab.ATTN_CAUSAL_TOP_LEFT)
    base.update(kw)
    return ab.sdpa_desc(**base)


def _status(ab, desc):
    f, b = C.c_size_t(), C.c_size_t()
    return ab._lib.load().sdpa_workspace_size(C.byref(desc), C.byref(f), C.byref(b)), b.value


def test_workspace_size(ab):
    st, nbytes = _status(ab, _desc(ab))
    assert st == 0
    t_pad = 4 * 1024  # each sequence rounded up to 128 rows
    assert nbytes >= 2 * 12 * t_pad * 4 + 12 * t_pad * 64 * 4
    st, det = _status(ab, _desc(ab, deterministic=True, dq_splits=4))
    assert st == 0 and det >= nbytes + 3 * 12 * t_pad * 64 * 4


def test_workspace_size_ordered(ab):
    """Ordered dQ mode: one accumulator plus one 32-bit counter per (head, 64 workspace rows)."""
    _, atomic = _status(ab, _desc(ab))
    st, ordered = _status(ab, _desc(ab, deterministic=ab.ATTN_DQ_ORDERED))
    assert st == 0 and ordered == atomic + 12 * (4 * 1024 // 64) * 4


def test_ordered_mode_unit_budget(ab):
    """Ordered dQ mode plans every work unit on the host: more than 4096 (key tiles of 128 x sequences
    x kv heads) is refused before any launch."""
    d = _desc(ab, b=64, h=32, h_kv=32, s_q=4096, s_kv=4096, d=128, deterministic=ab.ATTN_DQ_ORDERED)
    assert _bwd_call(ab, d) == 3
    assert _bwd_call(ab, _desc(ab, deterministic=ab.ATTN_DQ_ORDERED), ws=0) == 4  # within budget: next check


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), 2), (dict(h=12, h_kv=5), 2), (dict(b=0), 2), (dict(d=96), 3), (dict(d=256), 3),
    (dict(mask=5), 2), (dict(scale=float("nan")), 2), (dict(s_q=-1), 2), (dict(dq_splits=-2), 2),
    (dict(deterministic=3), 2), (dict(deterministic=-1), 2),
])
def test_descriptor_rejections(ab, kw, code):
    assert _status(ab, _desc(ab, **kw))[0] == code


def test_varlen_descriptor(ab):
    st, _ = _status(ab, _desc(ab, b=3, cu_seqlens_q=[10, 30, 60], cu_seqlens_kv=[10, 30, 60]))
    assert st == 0
    st, _ = _status(ab, _desc(ab, b=3, cu_seqlens_q=[10, 5, 60], cu_seqlens_kv=[10, 30, 60]))
    assert st == 2
    st, _ = _status(ab, _desc(ab, b=300, cu_seqlens_q=list(range(1, 301)), cu_seqlens_kv=list(range(1, 301))))
    assert st == 3


def _bwd_call(ab, desc, ptr=0x10000, stride=(8 * 1024 * 12 * 64, 64, 12 * 64), ws=0x100000, ws_bytes=1 << 40,
              lse=0x20000):
    v = ab.attn_view_t(ptr, *stride)
    return ab._lib.load().sdpa_bwd(C.byref(desc), v, v, v, v, v, C.cast(C.c_void_p(lse), C.POINTER(C.c_float)),
                                   v, v, v, C.c_void_p(ws), C.c_size_t(ws_bytes), None)


def test_bwd_rejects_before_launch(ab):
    d = _desc(ab)
    assert _bwd_call(ab, d, ptr=0) == 1                      # NULL tensor
    assert _bwd_call(ab, d, ptr=0x10008) == 5                # misaligned base
    assert _bwd_call(ab, d, stride=(8, 4, 64)) == 5          # stride not a multiple of 16 bytes
    assert _bwd_call(ab, d, ws=0) == 4                       # no workspace
    assert _bwd_call(ab, d, ws_bytes=100) == 4               # short workspace
    assert _bwd_call(ab, d, ws=0x100010) == 4                # misaligned workspace
    assert _bwd_call(ab, d, lse=0) == 1                      # no stats
    assert ab._lib.load().sdpa_bwd(None, *([ab.attn_view_t(0, 0, 0, 0)] * 5), None,
                                   *([ab.attn_view_t(0, 0, 0, 0)] * 3), None, 0, None) == 1


def _nsa(ab, **kw):
    base = dict(dtype=ab.ATTN_BF16, cu_seqlens_q=[4096, 8192], cu_seqlens_kv=[4096, 8192], n1=16, n2=1, d=128,
                scale=0.088, block_size=64, block_count=16, sparse_mode=2)
    base.update(kw)
    return ab.nsa_desc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(), 0), (dict(block_size=48), 2), (dict(block_size=256), 2), (dict(block_count=0), 2),
    (dict(block_count=128, block_size=64), 2), (dict(n1=16, n2=3), 2), (dict(n1=64, n2=1), 2),
    (dict(sparse_mode=1), 2), (dict(d=64), 2), (dict(d=192), 0), (dict(d_v=192), 0), (dict(d=192, d_v=128), 0),
    (dict(d_v=64), 2), (dict(grad_fp32=True), 0),
    (dict(cu_seqlens_kv=[4000, 8192]), 2), (dict(cu_seqlens_kv=[512, 1024], block_count=16), 2),
    (dict(deterministic=2), 0), (dict(deterministic=3), 2), (dict(deterministic=-1), 2),
])
def test_nsa_descriptor_rejections(ab, kw, code):
    n = C.c_size_t()
    assert ab._lib.load().nsa_workspace_size(C.byref(_nsa(ab, **kw)), C.byref(n)) == code


def test_nsa_ordered_workspace(ab):
    """Deterministic NSA modes: per-slot dQ partials (T1 n1 block_count d fp32) against one add counter per
    (token, kv head) (T1 n2 uint32) and an int32 per (token, kv head, slot) beside the single dQ
    accumulator; the first also keeps each work unit's dK / dV rows (block_size keys x (d + d_v) fp32) for
    a sum in unit order, for at most one unit per block-list row plus one per 32 chunks of 128 / R
    tokens."""
    lib = ab._lib.load()
    plain, split, ordered = C.c_size_t(), C.c_size_t(), C.c_size_t()
    assert lib.nsa_workspace_size(C.byref(_nsa(ab)), C.byref(plain)) == 0
    assert lib.nsa_workspace_size(C.byref(_nsa(ab, deterministic=1)), C.byref(split)) == 0
    assert lib.nsa_workspace_size(C.byref(_nsa(ab, deterministic=2)), C.byref(ordered)) == 0
    t1, n1, n2, cnt, d, bs, nrows = 8192, 16, 1, 16, 128, 64, 2 * 1 * 64
    align = lambda x: (x + 255) // 256 * 256
    tokens_per_unit = 32 * (128 // 16)  # G = 16: rows per token R = 16
    kv = align((nrows + -(-t1 * n2 * cnt // tokens_per_unit)) * bs * 2 * d * 4)
    assert split.value == plain.value + align(t1 * n1 * cnt * d * 4) + kv
    assert ordered.value == plain.value + align(t1 * n2 * 4) + align(t1 * n2 * cnt * 4)


def test_nsa_fwd_workspace_size(ab):
    """The tensor-core forward (d = d_v = 128, blocks of 64) uses the backward's workspace layout without
    deterministic partials; the CUDA-core forward (a head dim of 192) the status word alone."""
    lib = ab._lib.load()
    fwd, bwd = C.c_size_t(), C.c_size_t()
    assert lib.nsa_fwd_workspace_size(C.byref(_nsa(ab, deterministic=True)), C.byref(fwd)) == 0
    assert lib.nsa_workspace_size(C.byref(_nsa(ab)), C.byref(bwd)) == 0
    assert fwd.value == bwd.value
    assert lib.nsa_fwd_workspace_size(C.byref(_nsa(ab, d=192)), C.byref(fwd)) == 0 and fwd.value == 256


def test_nsa_fwd_rejects_before_launch(ab):
    lib = ab._lib.load()
    desc = _nsa(ab)
    n = C.c_size_t()
    assert lib.nsa_fwd_workspace_size(C.byref(desc), C.byref(n)) == 0 and n.value >= 4
    fp = lambda a: C.cast(C.c_void_p(a), C.POINTER(C.c_float))
    ip = lambda a: C.cast(C.c_void_p(a), C.POINTER(C.c_int32))

    def call(q=0x10000, o=0x30000, topk=0x40000, smax=0x50000, ws=0x100000, nbytes=256):
        return lib.nsa_selected_attn_fwd(C.byref(desc), C.c_void_p(q), C.c_void_p(0x10000), C.c_void_p(0x10000),
                                         ip(topk), C.c_void_p(o), fp(smax), fp(0x60000), C.c_void_p(ws),
                                         C.c_size_t(nbytes), None)
    assert call(q=0) == 1            # NULL query
    assert call(o=0x30008) == 5      # misaligned output
    assert call(topk=0x40002) == 5   # topk not 4-byte aligned
    assert call(smax=0x50004) == 5   # stats not 16-byte aligned
    assert call(nbytes=2) == 4       # short workspace
    assert call(ws=0) == 4           # no workspace


def test_fwd_rejects_before_launch(ab):
    lib = ab._lib.load()
    d = _desc(ab)
    v = ab.attn_view_t(0x10000, 8 * 1024 * 12 * 64, 64, 12 * 64)
    lse = C.cast(C.c_void_p(0x20000), C.POINTER(C.c_float))
    call = lambda view=v, lse=lse, ws=0x100000, nbytes=256: lib.sdpa_fwd_stats(
        C.byref(d), view, view, view, view, lse, C.c_void_p(ws), C.c_size_t(nbytes), None)
    assert call(lse=None) == 1                                               # no stats output
    assert call(view=ab.attn_view_t(0x10004, v.sb, v.sh, v.ss)) == 5        # misaligned base
    assert call(nbytes=16) == 4                                              # short workspace
    assert call(ws=0) == 4                                                   # no workspace


def test_nsa_bwd_rejects_before_launch(ab):
    lib = ab._lib.load()
    desc = _nsa(ab)
    n = C.c_size_t()
    assert lib.nsa_workspace_size(C.byref(desc), C.byref(n)) == 0
    fp = lambda a: C.cast(C.c_void_p(a), C.POINTER(C.c_float))
    ip = lambda a: C.cast(C.c_void_p(a), C.POINTER(C.c_int32))

    def call(q=0x10000, dq=0x30000, topk=0x40000, smax=0x50000, ws=0x100000, nbytes=None):
        t = [C.c_void_p(q)] + [C.c_void_p(0x10000)] * 4
        return lib.nsa_selected_attn_bwd(C.byref(desc), *t, fp(smax), fp(0x60000), ip(topk), C.c_void_p(dq),
                                         C.c_void_p(0x70000), C.c_void_p(0x80000), C.c_void_p(ws),
                                         C.c_size_t(n.value if nbytes is None else nbytes), None)
    assert call(q=0) == 1                 # NULL query
    assert call(dq=0x30008) == 5          # misaligned gradient
    assert call(topk=0x40002) == 5        # topk not 4-byte aligned
    assert call(smax=0x50004) == 5        # stats not 16-byte aligned
    assert call(nbytes=n.value - 1) == 4  # short workspace
    assert call(ws=0) == 4                # no workspace


def test_static_scratch_rejects_large_problems(ab):
    """A problem whose workspace exceeds the static scratch is refused before anything runs."""
    d = _desc(ab, b=2, h=32, h_kv=32, s_q=4096, s_kv=4096, d=128, dtype=ab.ATTN_BF16)
    v = ab.attn_view_t(0x10000, 4096 * 32 * 128, 128, 32 * 128)
    lse = C.cast(C.c_void_p(0x20000), C.POINTER(C.c_float))
    assert ab._lib.load().sdpa_bwd_static_scratch(C.byref(d), v, v, v, v, v, lse, v, v, v, None) == 4


def test_query_status_needs_its_pointers(ab):
    lib = ab._lib.load()
    flags = C.c_uint32()
    assert lib.attn_query_status(None, None, C.byref(flags)) == 1
    assert lib.attn_query_status(C.c_void_p(0x100000), None, None) == 1


def test_selftest_rejects_before_launch(ab):
    """The wait-timeout self-test checks its arguments on the host: no workspace, a short or
    misaligned one, and limits outside (0, 2] seconds launch nothing."""
    lib = ab._lib.load()
    call = lambda ws=0x100000, n=256, lim=0.02: lib.attn_selftest_wait_timeout(C.c_void_p(ws), C.c_size_t(n),
                                                                                 C.c_double(lim), None)
    assert call(ws=0) == 1
    assert call(n=2) == 4
    assert call(ws=0x100002) == 4
    assert call(lim=0.0) == 2
    assert call(lim=5.0) == 2
    assert call(lim=float("nan")) == 2


def test_occupy_rejects_before_launch(ab):
    lib = ab._lib.load()
    assert lib.attn_selftest_occupy(0, 1024, C.c_double(0.1), None) == 2
    assert lib.attn_selftest_occupy(8, 300 * 1024, C.c_double(0.1), None) == 2
    assert lib.attn_selftest_occupy(8, 1024, C.c_double(9.0), None) == 2
    assert lib.attn_selftest_occupy(8, 1024, C.c_double(0.0), None) == 2


def test_static_scratch_status_needs_its_pointer(ab):
    assert ab._lib.load().attn_static_scratch_status(None, None) == 1


def test_status_strings(ab):
    for code in range(8):
        assert ab._lib.load().attn_status_string(code).startswith(b"ATTN_")
