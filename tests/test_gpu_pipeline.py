"""The staged kernels' primitives on the GPU: a bulk (TMA) copy completes its
mbarrier with the right bytes, an arrival completes a phase, and a wait whose
phase nothing completes gives up after its 2-second bound and says so (the
failure path of the staged kernels' waits, made to run out without a fault:
the GPU stays usable, as the copy check run afterwards shows)."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("pipecheck") / "pipeline_check.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "adamw_update_gb300", "csrc"), "-Xcompiler", "-fPIC",
                    "-shared", os.path.join(ROOT, "tests", "cuda", "pipeline_check.cu"), "-o", out],
                   check=True)
    return ctypes.CDLL(out)


def _copy(lib, n):
    src = np.random.default_rng(n).integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    out = np.zeros(2 + n, np.uint64)
    assert lib.run_copy_check(src.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint32(n),
                              out.ctypes.data_as(ctypes.c_void_p)) == 0
    assert out[0] == 1
    assert np.array_equal(out[2:].astype(np.uint32), src)


@pytest.mark.parametrize("n", [4, 256, 1024])
def test_bulk_copy_completes_its_barrier(lib, n):
    _copy(lib, n)


def test_arrival_completes_a_phase(lib):
    out = np.zeros(2, np.uint64)
    assert lib.run_wait_check(0, out.ctypes.data_as(ctypes.c_void_p)) == 0
    assert out[0] == 1


def test_unfinished_phase_times_out_and_reports(lib):
    out = np.zeros(2, np.uint64)
    assert lib.run_wait_check(1, out.ctypes.data_as(ctypes.c_void_p)) == 0
    assert out[0] == 0  # gave up, reported, returned
    assert 2.0e9 <= out[1] < 10.0e9, out[1]  # after the 2 s bound, not forever
    _copy(lib, 64)  # the GPU is still usable
