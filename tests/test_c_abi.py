"""The C ABI from C: tests/c_abi_check.c is compiled with gcc against include/pgt.h and
linked to libpgt.so and the CUDA runtime; no Python in the caller's path."""
import os
import subprocess

import pytest

from persistent_gemm_tile_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    lib = _build.build()
    out = str(tmp_path_factory.mktemp("cabi") / "c_abi_check")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-O1", "-o", out, os.path.join(ROOT, "tests", "c_abi_check.c"),
           f"-I{ROOT}/include", f"-I{CUDA}/include", f"-L{libdir}", "-lpgt", f"-L{CUDA}/lib64", "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{CUDA}/lib64"]
    subprocess.run(cmd, check=True)
    return out


def test_c_caller_argument_checks(exe):
    r = subprocess.run([exe, "cpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "cpu checks: ok" in r.stdout


@pytest.mark.gpu
def test_c_caller_gemm_and_add_on_gpu(exe):
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gpu checks: ok" in r.stdout
