"""The C ABI used from a plain C program (gcc, no Python in the loop)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_roundtrip.c")
LIBDIR = os.path.join(ROOT, "async_bulk_tensor_gb300")
CUDA_LIB = "/usr/local/cuda/lib64"


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    import async_bulk_tensor_gb300  # noqa: F401  (fails loudly if libatb.so is missing)

    exe = tmp_path_factory.mktemp("c_abi") / "abi_roundtrip"
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"), SRC,
                           "-o", str(exe), "-L", LIBDIR, "-latb", "-L", CUDA_LIB, "-lcudart",
                           f"-Wl,-rpath,{LIBDIR}", f"-Wl,-rpath,{CUDA_LIB}"])
    return str(exe)


def test_c_program_host_checks(program):
    r = subprocess.run([program, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"


@pytest.mark.gpu
def test_c_program_round_trip_on_gpu(program):
    r = subprocess.run([program, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
