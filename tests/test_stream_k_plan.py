"""Host logic of the stream-K schedule, checked on the CPU.

tests/c/sk_plan_check.cu includes the kernel header and calls the very
functions that the host API (tg::sk_plan) and the kernel (tg::sk_bound,
tg::sk_owner, tg::sk_piece) use.  It replays every unit's work items for a
sweep of tile counts, unit counts and k-block counts, and checks that the
pieces partition each stream-K tile exactly once in slice order, that the
slabs they write lie inside the workspace, and that every whole tile has one
owner.  Compiled as host code with nvcc; no GPU is involved.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        pytest.skip("nvcc not available")
    return exe


def test_stream_k_pieces_partition_every_tile(tmp_path):
    exe = tmp_path / "sk_plan_check"
    cmd = [_nvcc(), "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "grouped_gemm_persistent_gb300", "csrc"), "-I", os.path.join(ROOT, "include"),
           "-o", str(exe), os.path.join(ROOT, "tests", "c", "sk_plan_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip().startswith("OK"), out.stdout
    _, plans, sk_plans, rasters = out.stdout.split()
    assert int(plans) > 30000 and int(sk_plans) > 10000     # the sweep exercised stream-K plans
    assert int(rasters) == 40 * 40 * 6
