"""A C program (tests/c/abi_example.c) built with gcc against include/basp.h
and libbasp.so, and a C++ one (tests/c/abi_example.cpp) against the C++ layer
include/basp.hpp: the ABI as C and C++ callers use it.  Host-only checks run
on the CPU; the GPU forms re-lay out cudaMalloc'd buffers and compare with
the C oracle."""
import os
import subprocess

import pytest

import oracle
from sequence_re_layout_gb300.build import LIB_PATH, build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path_factory, compiler, std, source, name):
    build_library()
    oracle_lib = oracle.build()
    exe = str(tmp_path_factory.mktemp("c") / name)
    libdir = os.path.dirname(LIB_PATH)
    odir = os.path.dirname(oracle_lib)
    cmd = [compiler, "-std=" + std, "-O1", "-o", exe, os.path.join(ROOT, "tests", "c", source),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-lbasp", "-L", odir, "-lbasp_oracle",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + odir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    return _build(tmp_path_factory, "gcc", "c11", "abi_example.c", "abi_example")


@pytest.fixture(scope="module")
def cpp_program(tmp_path_factory):
    return _build(tmp_path_factory, "g++", "c++17", "abi_example.cpp", "abi_example_cpp")


def test_c_program_host_checks(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi_example ok" in r.stdout


@pytest.mark.gpu
def test_c_program_on_gpu(program):
    r = subprocess.run([program, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "abi_example ok" in r.stdout


def test_cpp_layer_host_checks(cpp_program):
    r = subprocess.run([cpp_program], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi_example_cpp ok" in r.stdout


@pytest.mark.gpu
def test_cpp_layer_on_gpu(cpp_program):
    r = subprocess.run([cpp_program, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "abi_example_cpp ok" in r.stdout


def test_scratch_address_cache_follows_the_context(tmp_path):
    """The no-allocation entry point caches its scratch array's device address
    per CUDA context: a new context (as after a device reset) gets a fresh
    lookup, never the old address.  Host test with a fake context query."""
    exe = str(tmp_path / "scratch_cache_test")
    subprocess.run(["g++", "-std=c++17", "-O1", "-pthread", "-o", exe,
                    os.path.join(ROOT, "tests", "c", "scratch_cache_test.cpp"),
                    "-I", os.path.join(ROOT, "sequence_re_layout_gb300", "csrc")], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "scratch_cache ok" in r.stdout
