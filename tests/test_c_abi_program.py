"""A C program (tests/c/abi_example.c) built with gcc against include/basp.h
and libbasp.so: the C ABI as a C caller uses it.  Host-only checks run on the
CPU; the GPU form re-lays out cudaMalloc'd buffers and compares with the C
oracle."""
import os
import subprocess

import pytest

import oracle
from sequence_re_layout_gb300.build import LIB_PATH, build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    build_library()
    oracle_lib = oracle.build()
    exe = str(tmp_path_factory.mktemp("c") / "abi_example")
    libdir = os.path.dirname(LIB_PATH)
    odir = os.path.dirname(oracle_lib)
    cmd = ["gcc", "-std=c11", "-O1", "-o", exe, os.path.join(ROOT, "tests", "c", "abi_example.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-lbasp", "-L", odir, "-lbasp_oracle",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + odir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


def test_c_program_host_checks(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi_example ok" in r.stdout


@pytest.mark.gpu
def test_c_program_on_gpu(program):
    r = subprocess.run([program, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "abi_example ok" in r.stdout
