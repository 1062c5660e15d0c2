"""The step's zero-safe arithmetic against the plain IEEE arithmetic on the GPU.

Warps with an exactly-zero gradient divide v' by the bias correction with
Markstein's FMA correction of a quotient formed with the correctly rounded
reciprocal, and select the dividend for a zero update dividend.  Checked here:
the division against the IEEE divide __fdiv_rn for every dividend significand
with every 64th divisor significand (all 2^46 pairs with
PA_EXHAUSTIVE_DIVISION=1, about 45 s on a GB300), and whole elements
(adamw_element, zero-safe against plain) on 2^30 random elements whose
values, scalars and hyperparameters include zeros, subnormals, extremes, Inf
and NaN.  The per-vector path's branch-free arithmetic: the residual-corrected
square roots against __fsqrt_rn for every binary32 in [2^-100, 2^126) (and the
zero-safe one at +-0), and
adamw_vector (the warp's vote between the branch-free and the zero-safe
arithmetic) against adamw_element on 2^29 elements per bias-correction case,
with warps at the edges of the branch-free ranges; both arms must run."""
import ctypes
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("zscheck") / "step_division_check.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "adamw_update_gb300", "csrc"), "-Xcompiler", "-fPIC",
                    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-shared",
                    os.path.join(ROOT, "tests", "cuda", "step_division_check.cu"), "-o", out],
                   check=True)
    return ctypes.CDLL(out)


def test_division_by_reciprocal_equals_ieee(lib):
    step = 1 if os.environ.get("PA_EXHAUSTIVE_DIVISION") == "1" else 64
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    assert lib.run_significands(ctypes.c_uint32(step), ctypes.byref(count), first) == 0
    assert count.value == 0, (count.value, [hex(x) for x in first])


def test_zero_safe_element_equals_plain(lib):
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    assert lib.run_elements(ctypes.c_uint64(1 << 30), ctypes.c_uint64(17), ctypes.byref(count),
                            first) == 0
    assert count.value == 0, (count.value, [hex(x) for x in first])


def test_residual_root_equals_ieee_on_its_range(lib):
    count = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    assert lib.run_roots(ctypes.byref(count), first) == 0
    assert count.value == 0, (count.value, [hex(x) for x in first])


@pytest.mark.parametrize("paired", [0, 1])
@pytest.mark.parametrize("unit_bc2", [0, 1])
def test_vector_arithmetic_equals_element(lib, unit_bc2, paired):
    nwarps = 1 << 22
    count = ctypes.c_ulonglong(0)
    branch_free = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 4)()
    assert lib.run_vectors(ctypes.c_int(unit_bc2), ctypes.c_int(paired), ctypes.c_uint64(nwarps),
                           ctypes.c_uint64(23), ctypes.byref(count), first,
                           ctypes.byref(branch_free)) == 0
    assert count.value == 0, (count.value, [hex(x) for x in first])
    # both arms ran: about half of the warps are drawn in range
    assert nwarps // 5 < branch_free.value < nwarps * 4 // 5, branch_free.value
