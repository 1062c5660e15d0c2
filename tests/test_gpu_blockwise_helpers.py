"""The blockwise requantiser's fast helpers against their plain forms on the
GPU (KBench "quantized-optimizer-state" reference.py, _requantise): the bucket
table search equals the binary search over the 255 midpoints for every
binary32 c in [-1, 1] (exhaustive, three maps), and the FMA division by the
block scale (Markstein's correction with the correctly rounded reciprocal)
equals the IEEE quotient __fdiv_rn on 4e9 random (x, scale) pairs with
|x| <= scale, zeros and subnormal x included; the Newton-refined reciprocal
equals __frcp_rn for every scale of the fast range [2^-100, 2^100); and whole
codes as the requantiser forms them (that reciprocal, the FMA quotient, the
bucket search, the IEEE fix-up below the floor) equal
the count of midpoints below the IEEE quotient on 2^30 random pairs per map."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("bwcheck") / "blockwise_check.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "adamw_update_gb300", "csrc"), "-Xcompiler", "-fPIC",
                    "-shared", os.path.join(ROOT, "tests", "cuda", "blockwise_check.cu"), "-o", out],
                   check=True)
    return ctypes.CDLL(out)


@pytest.mark.parametrize("kind", ["dynamic_signed", "dynamic_unsigned", "linear", "random"])
def test_bucket_search_equals_binary_search_everywhere(lib, kind):
    q = {"dynamic_signed": wl.dynamic_qmap_signed, "dynamic_unsigned": wl.dynamic_qmap_unsigned,
         "linear": wl.linear_qmap_signed, "random": lambda: wl.random_qmap(7, True)}[kind]()
    q = np.ascontiguousarray(q, np.float32)
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    rc = lib.run_search_all(q.ctypes.data_as(ctypes.c_void_p), ctypes.byref(count), first)
    assert rc == 0
    assert count.value == 0, (kind, count.value, list(first))


def test_block_division_equals_ieee(lib):
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    rc = lib.run_divide_random(ctypes.c_uint64(4 << 30), ctypes.c_uint64(99), ctypes.byref(count), first)
    assert rc == 0
    assert count.value == 0, (count.value, [hex(x) for x in first])


def test_reciprocal_equals_ieee_on_the_fast_range(lib):
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    assert lib.run_reciprocal_all(ctypes.byref(count), first) == 0
    assert count.value == 0, (count.value, [hex(x) for x in first])


@pytest.mark.parametrize("kind", ["dynamic_signed", "dynamic_unsigned", "linear", "random"])
def test_requantised_codes_equal_the_ieee_definition(lib, kind):
    q = {"dynamic_signed": wl.dynamic_qmap_signed, "dynamic_unsigned": wl.dynamic_qmap_unsigned,
         "linear": wl.linear_qmap_signed, "random": lambda: wl.random_qmap(7, True)}[kind]()
    q = np.ascontiguousarray(q, np.float32)
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    rc = lib.run_codes_random(q.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(1 << 30),
                              ctypes.c_uint64(5), ctypes.byref(count), first)
    assert rc == 0
    assert count.value == 0, (kind, count.value, [hex(x) for x in first])
