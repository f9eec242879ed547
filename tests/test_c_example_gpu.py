"""The library used from plain C99 with the CUDA runtime's C API (no Python,
no torch): tests/c/gemm_example.c is compiled with gcc, linked against
libtcgemm.so and libcudart, run, and must report every element exact."""
import os
import shutil
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_c_program_runs_a_gemm(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    from tiled_tensor_core_persistent_gb300 import _build
    so = _build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                           os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib")) if os.path.isdir(d)]
    exe = tmp_path / "gemm_example"
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "gemm_example.c"), "-o", str(exe),
           so, f"-Wl,-rpath,{os.path.dirname(so)}"]
    for d in libdirs:
        cmd += [f"-L{d}", f"-Wl,-rpath,{d}"]
    cmd += ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "every element exact" in r.stdout
