"""The C ABI from plain C: tests/c/tg_c_client.c is compiled against include/tg.h
and libtg.so with gcc (CPU: it must build), and run on the GPU (exact integer
results compared element by element by the program itself)."""
import os
import shutil
import subprocess

import pytest

from grouped_gemm_persistent_gb300 import _binding
from grouped_gemm_persistent_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path):
    build()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = os.path.join(tmp_path, "tg_c_client")
    libdir = os.path.dirname(_binding.LIB_PATH)
    cmd = [gcc, "-O1", "-std=c99", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c", "tg_c_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-ltg", "-Wl,-rpath," + libdir,
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_builds(tmp_path):
    _compile(str(tmp_path))


@pytest.mark.gpu
def test_c_client_runs(tmp_path):
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 mismatches" in r.stdout and "ok" in r.stdout
