"""The C ABI used from a plain C99 program (tests/c_abi/abi_check.c).

The program includes only include/*.h and links only libpurlin.so and the CUDA
runtime.  On the CPU it plans an AllGather (host-only call); on the GPU it runs
an AllReduce and a ReduceScatter + AllGather of fp32 integers and checks the
exact sums it computes itself, and times the host side of small AllReduces.
"""
import json
import os
import shutil
import subprocess

import pytest

import reduce_datapath_gb300 as rd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    from reduce_datapath_gb300 import _build
    return os.path.dirname(os.path.dirname(_build.nvcc()))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    rd.build()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    exe = str(tmp_path_factory.mktemp("c_abi") / "abi_check")
    libdir = os.path.dirname(rd.LIB_PATH)
    cmd = [gcc, "-std=c99", "-O1", "-Wall", "-Werror", "-o", exe,
           os.path.join(ROOT, "tests", "c_abi", "abi_check.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-lpurlin", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_plan_from_c(program):
    r = subprocess.run([program, "plan"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_collectives_from_c(program):
    r = subprocess.run([program, "gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_host_cost_from_c(program):
    """Host time per call of a 4 KiB-per-rank AllReduce from C: one JSON line,
    planning far below the launch (loose bounds: a shared host)."""
    r = subprocess.run([program, "cost"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    cost = json.loads(r.stdout.strip().splitlines()[-1])
    assert cost["segments"] == 1
    assert 0 < cost["plan_segments_us"] < 20
    assert 0 < cost["record_plan_us"] < 50
    assert 0 < cost["plan_launch_us"] < 200 and 0 < cost["call_us"] < 200
