"""The C ABI on the CPU (no GPU needed): libpackedadam.so loads and exports
every function include/packedadam.h declares, host-side argument checks
return their documented status before anything touches CUDA, and the oracle
and the CUDA path share no source."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "packedadam.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_pa_build", os.path.join(ROOT, "adamw_update_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    try:
        mod.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    import adamw_update_gb300 as pa

    return pa


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ("pa_encode_state", "pa_decode_state", "pa_adamw_step_packed_e4",
                 "pa_adamw_step_fp32", "pa_adamw_step_packed_fp16", "pa_adamw_step_blockwise8",
                 "pa_adamw_step_packed_e4_multi", "pa_version", "pa_status_string"):
        assert want in names, want


@pytest.mark.parametrize("variant", [False, True], ids=["exact", "fast"])
def test_library_exports_every_declared_symbol(lib, variant):
    so = ctypes.CDLL(lib.library_path(fast=variant))
    missing = [n for n in _declared() if not hasattr(so, n)]
    assert not missing, missing


def test_binding_names_match_the_abi(lib):
    for name in _declared():
        if name in ("pa_last_error",):
            continue
        assert hasattr(lib, name), name


def test_host_validation_without_gpu(lib):
    L = lib._lib
    hy = (1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert L.pa_version() == 10000
    assert L.pa_status_string(0) == b"PA_OK"
    assert L.pa_adamw_step_packed_e4(None, None, None, 4, 0, *hy, None, None) == 2  # step < 1
    assert L.pa_adamw_step_packed_e4(None, None, None, 4, 1, 1e-3, 1.0, 0.999, 1e-8, 0.0,
                                     None, None) == 2  # beta1 = 1
    assert L.pa_adamw_step_packed_e4(None, None, None, 4, 1, float("inf"), 0.9, 0.999, 1e-8,
                                     0.0, None, None) == 2
    assert L.pa_adamw_step_packed_e4(None, None, None, 4, 1, 1e-3, 0.9, 0.999, -1.0, 0.0,
                                     None, None) == 2  # eps < 0
    assert L.pa_adamw_step_packed_e4(None, None, None, -1, 1, *hy, None, None) == 2
    assert L.pa_adamw_step_packed_e4(None, None, None, 4, 1, *hy, None, None) == 1
    assert L.pa_adamw_step_packed_e4(None, None, None, 0, 1, *hy, None, None) == 0
    L.pa_adamw_step_packed_e4(None, None, None, 4, 0, *hy, None, None)
    assert b"step" in L.pa_last_error()
    bad = ctypes.c_void_p(0x1002)  # never dereferenced: rejected as misaligned first
    assert L.pa_adamw_step_packed_e4(bad, bad, bad, 4, 1, *hy, None, None) == 3
    assert L.pa_adamw_step_fp32(bad, bad, bad, None, 4, 1, *hy, None, None) == 1
    assert L.pa_adamw_step_packed_e4_multi(None, -1, 1, *hy, None, None) == 2
    assert L.pa_adamw_step_packed_e4_multi(None, 0, 1, *hy, None, None) == 0
    assert L.pa_adamw_step_packed_e4_multi(None, 3, 1, *hy, None, None) == 1
    t = (lib.PaTensor * 2)(lib.PaTensor(0x1000, 0x2000, 0x3000, None, -5), lib.PaTensor())
    assert L.pa_adamw_step_packed_e4_multi(t, 2, 1, *hy, None, None) == 2
    assert b"tensor 0" in L.pa_last_error()
    # a one-tensor list (passed by value, no table) is checked like any list
    one = (lib.PaTensor * 1)(lib.PaTensor(0x1000, 0x2000, 0x3000, None, -5))
    assert L.pa_adamw_step_packed_e4_multi(one, 1, 1, *hy, None, None) == 2
    assert b"tensor 0" in L.pa_last_error()
    one = (lib.PaTensor * 1)(lib.PaTensor(0x1002, 0x2000, 0x3000, None, 4))
    assert L.pa_adamw_step_packed_e4_multi(one, 1, 1, *hy, None, None) == 3
    assert L.pa_adamw_step_fp32_multi(one, 1, 1, *hy, None, None) == 1  # no v
    one = (lib.PaTensor * 1)(lib.PaTensor(0x1000, 0x2000, 0x3000, None, 0))
    assert L.pa_adamw_step_packed_fp16_multi(one, 1, 1, *hy, None, None) == 0  # empty: no-op
    al = ctypes.c_void_p(0x1000)
    assert L.pa_adamw_step_blockwise8(al, ctypes.c_void_p(0x1004), al, al, al, al, al, al, al,
                                      4, 1, *hy, None, None) == 3  # g not 16-byte aligned
    assert L.pa_encode_state(None, None, None, 0, None, None) == 0
    assert L.pa_decode_state(None, None, None, 3, None) == 1
    # the TurboAdam-style step
    T = lib.PaTurboState
    st = T(0x1000, 0x2000, 0x3000, 0x4000, 0x5000)
    sd = (1.1, ctypes.c_uint64(7), None, None)
    assert L.pa_turbo_step(al, al, 4, ctypes.byref(st), 1, 1e-3, 0.9, 0.8, 1e-8, 0.0, *sd) == 2
    assert b"beta1^2 < beta2" in L.pa_last_error()
    assert L.pa_turbo_step(al, al, -1, ctypes.byref(st), 1, *hy, *sd) == 2
    assert L.pa_turbo_step(al, al, 4, ctypes.byref(st), 1 << 22, *hy, *sd) == 2
    assert L.pa_turbo_step(al, al, 4, ctypes.byref(st), 1, *hy, 0.0, ctypes.c_uint64(7), None,
                           None) == 2  # scale factor
    assert L.pa_turbo_step(al, al, 0, None, 1, *hy, *sd) == 0  # empty: no-op
    assert L.pa_turbo_step(al, al, 4, None, 1, *hy, *sd) == 1
    assert L.pa_turbo_step(ctypes.c_void_p(0x1004), al, 4, ctypes.byref(st), 1, *hy, *sd) == 3
    odd = T(0x1000, 0x2001, 0x3000, 0x4000, 0x5000)
    assert L.pa_turbo_step(al, al, 4, ctypes.byref(odd), 1, *hy, *sd) == 3


def test_oracle_and_cuda_path_share_no_source():
    """Neither side includes, imports or links the other."""
    cuda_dir = os.path.join(ROOT, "adamw_update_gb300")
    for dirpath, _, files in os.walk(cuda_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text.replace("the oracle", "")), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "adamw_update_gb300" not in text and "packedadam.h" not in text, f
            assert "codecs.cuh" not in text, f
