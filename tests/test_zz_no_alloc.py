"""The multi-tensor packed-E4 step that allocates nothing.

pa_adamw_step_packed_e4_multi_noalloc serves callers that cannot let a library
call cudaMalloc -- a framework whose caching allocator owns the device memory,
or a loop that must not meet cudaMalloc's implicit synchronisation.  It keeps
its descriptor table in a fixed device array instead.  Here it is called
through the C ABI and compared, bit for bit (the tolerance of every parity test
of this suite), with pa_adamw_step_packed_e4_multi on two calls in a row, and
with the CPU oracle on lists that fill the array's two upload batches: 600
ragged tensors and exactly 1024.  This file is collected last, so a run that
stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_same_bits, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu


def _noalloc_fn(pa):
    lib = ctypes.CDLL(pa.library_path())
    fn = lib.pa_adamw_step_packed_e4_multi_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(pa.PaTensor), ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                   ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                   ctypes.c_void_p, ctypes.c_void_p]
    return fn


def test_noalloc_step_matches_the_allocating_step_on_two_calls():
    import torch

    import adamw_update_gb300 as pa

    fn = _noalloc_fn(pa)
    sizes = [5, 0, 4096, 1, 30_001, 2048 * 3 + 7]
    rng = np.random.default_rng(41)
    a_p, a_s, b_p, b_s, grads = [], [], [], [], []
    for k, n in enumerate(sizes):
        off = k % 4  # views at every 4-byte phase
        p = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).cuda()
        s = torch.from_numpy(rng.integers(0, 1 << 31, n).astype(np.int32)).cuda()
        for dst, src in ((a_p, p), (b_p, p), (a_s, s), (b_s, s)):
            buf = torch.zeros(n + 8, dtype=src.dtype, device="cuda")
            view = buf[off:off + n]
            view.copy_(src)
            dst.append(view)
        grads.append(torch.zeros(n, dtype=torch.float32, device="cuda"))
    bad_a = torch.zeros(1, dtype=torch.int64, device="cuda")
    bad_b = torch.zeros(1, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    hy = wl.HYPER
    for t in (1, 2):
        for g in grads:
            g.copy_(torch.from_numpy(rng.normal(0, 1e-3, g.numel()).astype(np.float32)))
        grads[0][1] = float("nan")  # a counted non-finite element
        arr_a = pa.tensor_list(list(zip(a_p, grads, a_s)))
        rc = fn(arr_a, len(arr_a), t, hy["lr"], hy["beta1"], hy["beta2"], hy["eps"], hy["wd"],
                bad_a.data_ptr(), stream)
        assert rc == 0, pa._lib.pa_last_error()
        pa.pa_adamw_step_packed_e4_multi(list(zip(b_p, grads, b_s)), t, nonfinite=bad_b, **hy)
        torch.cuda.synchronize()
        for k in range(len(sizes)):
            pa_bits = a_p[k].view(torch.int32)
            pb_bits = b_p[k].view(torch.int32)
            assert torch.equal(pa_bits, pb_bits), f"p of tensor {k}, call {t}"
            assert torch.equal(a_s[k], b_s[k]), f"state of tensor {k}, call {t}"
        assert int(bad_a.item()) == int(bad_b.item()) == t


def test_noalloc_rejects_lists_beyond_its_array():
    import adamw_update_gb300 as pa

    fn = _noalloc_fn(pa)
    arr = (pa.PaTensor * 1025)()
    rc = fn(arr, 1025, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, None, None)
    assert rc == 2
    assert b"1024" in pa._lib.pa_last_error()


@pytest.mark.parametrize("count", [600, 1024])
def test_noalloc_long_lists_equal_the_oracle(count):
    """600 ragged tensors (past the 512 descriptors of one upload launch and of
    the kernel's shared-memory copy, so the walk reads the array in global
    memory) and exactly the array's 1024: two calls in a row, equal to the
    oracle and to the allocating step, bit for bit."""
    import torch

    import adamw_update_gb300 as pa

    fn = _noalloc_fn(pa)
    rng = np.random.default_rng(50 + count)
    sizes = [int(x) for x in rng.choice([0, 1, 3, 4, 7, 100, 6143, 6144, 6149, 12_300], count)]
    host_p = [rng.normal(0, 0.02, n).astype(np.float32) for n in sizes]
    host_s = [np.zeros(n, np.uint32) for n in sizes]
    views = []
    for k, n in enumerate(sizes):
        off = (k // 3) % 4  # views at every 4-byte phase
        pair = []
        for a, dt in ((host_p[k], torch.float32), (host_s[k], torch.int32)):
            buf = torch.zeros(n + 8, dtype=dt, device="cuda")
            v = buf[off:off + n]
            if n:
                v.copy_(dev(a))
            pair.append(v)
        views.append(pair)
    twin = [[v.clone() for v in pair] for pair in views]
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    hy = wl.HYPER
    for t in (1, 2):
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n in sizes]
        dgs = [dev(g) for g in gs]
        arr = pa.tensor_list([(v[0], g, v[1]) for v, g in zip(views, dgs)])
        rc = fn(arr, len(arr), t, hy["lr"], hy["beta1"], hy["beta2"], hy["eps"], hy["wd"],
                bad.data_ptr(), stream)
        assert rc == 0, pa._lib.pa_last_error()
        pa.pa_adamw_step_packed_e4_multi([(v[0], g, v[1]) for v, g in zip(twin, dgs)], t, **hy)
        for k, g in enumerate(gs):
            host_p[k], host_s[k], _ = oracle.step_packed(host_p[k], g, host_s[k], t, **hy)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
    for k in range(count):
        assert_same_bits(host_f32(views[k][0]), host_p[k], f"tensor {k} p")
        assert_same_bits(host_u32(views[k][1]), host_s[k], f"tensor {k} state")
        assert torch.equal(views[k][0].view(torch.int32), twin[k][0].view(torch.int32))
        assert torch.equal(views[k][1], twin[k][1])
