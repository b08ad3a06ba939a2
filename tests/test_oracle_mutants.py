"""The oracle's pins have teeth: plant plausible mistakes in copies of the
oracle source (CPU only), rebuild, and check that a pin fails for each."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, original text, mutated text, pin that must fail)
MUTANTS = [
    ("ds_sign", "const double ds = p * (dp - Di);", "const double ds = p * (dp + Di);", "dense_fd"),
    ("ds_dropped_D", "const double ds = p * (dp - Di);", "const double ds = p * dp;", "dense_fd"),
    ("dk_no_scale", "dkj[x] += pb->scale * ds * qi[x];", "dkj[x] += ds * qi[x];", "dense_fd"),
    ("dp_transposed_operand", "const double dp = dot(doi, vj, d);", "const double dp = dot(doi, kj, d);",
     "dense_fd"),
    ("causal_off_by_one", "if (mask == 1) return j <= i;", "if (mask == 1) return j < i;", "mask_bitmap"),
    ("bottom_right_shift", "if (mask == 2) return j <= i + (lkv - lq);",
     "if (mask == 2) return j <= i + (lq - lkv);", "mask_bitmap"),
    ("nsa_scatter_index", "c->dk[((k0 + rows[r]) * pb->n2 + g) * d + x] += dksel[r * d + x];",
     "c->dk[((k0 + r) * pb->n2 + g) * d + x] += dksel[r * d + x];", "nsa_fd"),
    ("nsa_sum_ignored", "const double p = exp(pb->scale * dot(qi, ksel + r * d, d) - mx) / sm;",
     "const double p = exp(pb->scale * dot(qi, ksel + r * d, d) - mx);", "nsa_fd"),
    ("dq_no_scale", "dqi[x] += pb->scale * ds * kj[x];", "dqi[x] += ds * kj[x];", "dense_fd"),
    ("dv_from_q", "dvj[x] += p * doi[x];", "dvj[x] += p * qi[x];", "dense_fd"),
    ("lse_without_max", "const double lse = mx + log(sum);", "const double lse = log(sum);", "two_keys"),
    # query heads of a kv head taken interleaved (h_kv apart) instead of contiguous, in the forward only
    ("gqa_interleaved", "for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {",
     "for (int64_t hq = g; hq < pb->h; hq += pb->h_kv) {", "dense_fd_gqa"),
    ("seq_boundary", "if (t < cu[b]) return b;", "if (t <= cu[b]) return b;", "sampled_rows"),
    ("nsa_block_offset", "rows[n++] = blk * pb->block_size + r;", "rows[n++] = blk + r;", "nsa_vs_dense"),
    ("nsa_D_from_dO", "const double mx = c->mx[row], sm = c->sm[row];\n            const double Di = dot(doi, oi, e);",
     "const double mx = c->mx[row], sm = c->sm[row];\n            const double Di = dot(doi, doi, e);", "nsa_fd"),
    # the value head dim mistaken for the query / key one (d < d_v in the pin, so reads stay in bounds)
    ("nsa_D_over_qk_dim", "const double mx = c->mx[row], sm = c->sm[row];\n            const double Di = dot(doi, oi, e);",
     "const double mx = c->mx[row], sm = c->sm[row];\n            const double Di = dot(doi, oi, d);", "nsa_fd_dims"),
    ("nsa_dv_scatter_stride", "c->dv[((k0 + rows[r]) * pb->n2 + g) * e + x] += dvsel[r * e + x];",
     "c->dv[((k0 + rows[r]) * pb->n2 + g) * d + x] += dvsel[r * e + x];", "nsa_fd_dims"),
    ("nsa_dk_no_scale", "dksel[r * d + x] += pb->scale * ds * qi[x];", "dksel[r * d + x] += ds * qi[x];",
     "nsa_fd"),
    ("block_lists_last_key", "nsa_mode_visible(pb, i, blk * pb->block_size, lq, lkv)",
     "nsa_mode_visible(pb, i, blk * pb->block_size + pb->block_size - 1, lq, lkv)", "block_lists"),
    # attenMaskOptional read as "keep" instead of "remove", and ignored altogether
    ("mask_inverted", "return !(pb->atten_mask && pb->atten_mask[i * pb->mask_cols + j]);",
     "return !(pb->atten_mask && !pb->atten_mask[i * pb->mask_cols + j]);", "mask_one_key"),
    ("mask_ignored", "return !(pb->atten_mask && pb->atten_mask[i * pb->mask_cols + j]);", "return 1;",
     "mask_causal"),
    ("repeat_accepted", "if (topk_tg[e] == blk) return -1;", "if (topk_tg[e] == blk && 0) return -1;", "nsa_repeat"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-pthread",
                           "-D_POSIX_C_SOURCE=200809L", "-o", str(so), str(path), "-lm"])
    return ctypes.CDLL(str(so))


def _run_pin(pin):
    if pin == "dense_fd":
        pins._check_dense_fd([5], [7], h=2, h_kv=1, d=3, scale=0.7, mask=oracle.CAUSAL_BOTTOM_RIGHT, seed=3)
    elif pin == "mask_bitmap":
        for mask, key in ((oracle.CAUSAL_TOP_LEFT, "top_left"), (oracle.CAUSAL_BOTTOM_RIGHT, "bottom_right")):
            pins.test_mask_bitmaps(mask, key)
    elif pin == "nsa_fd":
        pins.test_nsa_finite_differences(0)
    elif pin == "two_keys":
        pins.test_two_keys_closed_form()
    elif pin == "dense_fd_gqa":
        pins.test_dense_finite_differences_varlen_gqa(oracle.MASK_NONE)
    elif pin == "sampled_rows":
        pins.test_sampled_rows_equal_full()
    elif pin == "nsa_vs_dense":
        pins.test_nsa_gather_equals_masked_dense(0)
    elif pin == "block_lists":
        pins.test_nsa_block_lists_definition(2)
    elif pin == "nsa_repeat":
        pins.check_nsa_rejects_repeated_index()
    elif pin == "nsa_fd_dims":
        pins.test_nsa_finite_differences_unequal_dims(2)
    elif pin == "mask_one_key":
        pins.test_nsa_mask_keeps_one_key_closed_form()
    elif pin == "mask_causal":
        pins.test_nsa_causal_mask_equals_sparse_mode_2()
    else:
        raise ValueError(pin)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_mutant(tmp_path, monkeypatch, name, old, new, pin):
    _run_pin(pin)  # the real oracle passes this pin
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, name, old, new))
    with pytest.raises(AssertionError):
        _run_pin(pin)
