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


def test_struct_layouts_agree_with_the_c_compiler(exe):
    import ctypes

    import persistent_gemm_tile_gb300 as pgt
    out = subprocess.run([exe, "cpu"], capture_output=True, text=True, timeout=120).stdout
    lines = {ln.split()[1]: ln.split()[2:] for ln in out.splitlines() if ln.startswith("layout ")}
    desc = lines["pgt_gemm_desc"]
    c_layout = {"size": int(desc[0])}
    c_layout.update({desc[i]: int(desc[i + 1]) for i in range(1, len(desc), 2)})
    py = {"size": ctypes.sizeof(pgt.GemmDesc)}
    py.update({f: getattr(pgt.GemmDesc, f).offset for f in ("dtype", "ws_groups", "epilogue", "alpha", "ws_layout",
                                                            "bias")})
    assert py == c_layout
    other = lines["pgt_gemm_plan_info"]
    assert int(other[0]) == ctypes.sizeof(pgt.PlanInfo)
    assert int(other[2]) == ctypes.sizeof(pgt.Trace)
    assert int(other[4]) == ctypes.sizeof(pgt.ScaleSpace)


@pytest.mark.gpu
def test_c_caller_gemm_and_add_on_gpu(exe):
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gpu checks: ok" in r.stdout
