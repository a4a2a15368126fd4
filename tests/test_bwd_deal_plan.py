"""The host side of the backward's dealt causal launches, checked without a GPU:
tests/host/deal_plan_check.cu includes the backward's source, asks it for the
per-CTA lists of causal problems of many shapes (batch, query and key/value
heads, ragged and long sequences) on 152 SMs, and checks that every key-tile
item appears exactly once, whole or as both of its two parts, that the lists are
ordered and fit the table, that parts use only the workspace's partial slots
and counters, and that no split item has fewer than two steps.  A dropped or doubled item would otherwise only show as wrong
gradients for the shapes the GPU tests happen to run."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_52_gb300", "csrc")


def test_deal_lists_cover_every_item_once(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "deal_plan_check")
    # device code as PTX only (no GPU code generation needed: nothing is launched)
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=compute_103a",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    os.path.join(ROOT, "tests", "host", "deal_plan_check.cu"), "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
