"""The C ABI from C alone: tests/c/abi_smoke.c is compiled as strict C11
against include/tiled_gemm.h and linked to the library (CPU: the header is
plain C and every call it makes resolves), then run on the GPU, where it
checks gemm, gemm_ex and gemm_general against an integer loop on the host."""
import os
import shutil
import subprocess

import pytest

import tiled_matrix_multiplication_output_gb300 as tg
from tiled_matrix_multiplication_output_gb300 import build as tg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_smoke.c")


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(tg_build.LIB_PATH):
        pytest.skip("library not built")
    cuda = _cuda_home()
    lib_dir = os.path.dirname(tg_build.LIB_PATH)
    exe = os.path.join(out_dir, "abi_smoke")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), SRC,
           "-L", lib_dir, "-ltiled_gemm", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_is_c11_and_links(tmp_path):
    _compile(str(tmp_path))


@pytest.mark.gpu
def test_c_program_multiplies_exactly(tmp_path):
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
