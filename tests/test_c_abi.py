"""libep from plain C: tests/c_abi/abi_check.c includes only include/ep.h
and the CUDA runtime, drives the low-latency and normal paths with
cudaMalloc'd buffers and compares every result with the C oracle.  Built
here (gcc) to show the header is a C header and the program links; run on
a GPU."""
import os
import shutil
import subprocess

import pytest

from combine_get_dispatch_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build_program(out_dir):
    import oracle
    lib = _build.build()
    olib = oracle.build()
    exe = os.path.join(out_dir, "abi_check")
    libdir, olibdir = os.path.dirname(lib), os.path.dirname(olib)
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Werror", "-Wno-unused-variable",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_check.c"),
           "-L", libdir, "-lep", "-L", olibdir, "-lep_oracle",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{olibdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}",
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_builds_against_the_header(tmp_path):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    assert os.path.exists(_build_program(str(tmp_path)))


@pytest.mark.gpu
def test_c_program_matches_the_oracle(tmp_path):
    exe = _build_program(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi check ok" in r.stdout
