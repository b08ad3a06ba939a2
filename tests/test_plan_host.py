"""The dense backward's host plans (bwd_tc.cu, plan_units / plan_ordered), run on the CPU: a host
program built with nvcc plans the benchmark shapes and some edge shapes in the atomic, split and
ordered dQ modes.  Every plan must end, take every unit with work exactly once, and in the ordered
mode give each CTA its units in non-increasing key-tile order (the condition under which its waits
cannot form a cycle); the NSA ordered mode's unit order is checked the same way."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_backward_02_gb300", "csrc")


@pytest.fixture(scope="module")
def plan_lines():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "plan_check")
        subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-O1", "-gencode",
                        "arch=compute_103a,code=sm_103a", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                        os.path.join(ROOT, "tests", "plan_check.cu"), "-o", exe],
                       check=True, capture_output=True, timeout=600)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout
    lines = {}
    for line in out.splitlines():
        f = line.split()
        lines[f[0]] = {k: int(v) for k, v in zip(f[1::2], f[2::2])}
    return lines


def test_every_shape_planned(plan_lines):
    dense = {k: v for k, v in plan_lines.items() if not k.startswith("nsa_order")}
    assert len(dense) == 15
    for name, r in dense.items():
        if name.startswith("varlen") and name.endswith("_split"):
            assert r["on"] in (0, 1), name  # packed split batches may keep the snake order
        if r["on"]:
            assert r["planned"] == r["work"], (name, r)
            assert r["twice"] == 0, (name, r)


def test_fixed_length_batches_are_planned(plan_lines):
    for name in ("w1_atomic", "w2_atomic", "ragged_gqa_atomic", "w1_ordered", "w2_ordered"):
        assert plan_lines[name]["on"] == 1, name


def test_ordered_lists_take_key_tiles_in_decreasing_order(plan_lines):
    for name, r in plan_lines.items():
        if name.endswith("_ordered"):
            assert r["on"] == 1 and r["ordered_ok"] == 1, (name, r)


def test_nsa_ordered_unit_order(plan_lines):
    """NSA ordered deterministic mode: the rows in decreasing block order form a permutation and the blocks
    never increase along it."""
    rows = {k: v for k, v in plan_lines.items() if k.startswith("nsa_order")}
    assert len(rows) == 3
    for name, r in rows.items():
        assert r["perm"] == 1 and r["mono"] == 1, (name, r)
