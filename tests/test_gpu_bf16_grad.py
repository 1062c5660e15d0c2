"""Packed-E4 steps that read bfloat16 gradients: bit for bit equal to the
oracle run on the exactly widened gradient, single tensors and lists: views
whose gradient is 16-byte aligned where p's 16-byte body starts (staged, with
and without a head peel: offsets (0,0,0), (1,5,1), (3,7,3)), views where it is
only 8-byte aligned there, and mismatched phases (the 4-byte path)."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_same_bits, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu
HY = wl.HYPER


def _bf16(rng, n):
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    bits = (g.view(np.uint32) >> 16).astype(np.uint16)  # truncation is fine: any bf16 input
    return bits, (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n", [1, 7, 4096, 4099, 12_300, 70_001])
@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 5, 1), (3, 7, 3), (1, 1, 1), (3, 3, 3),
                                     (1, 2, 1)])
def test_single_bf16_gradient(n, offsets):
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(n + sum(offsets))
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = np.zeros(n, np.uint32)
    bp = torch.zeros(n + 8, dtype=torch.float32, device="cuda")
    bg = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    bs = torch.zeros(n + 8, dtype=torch.int32, device="cuda")
    dp, dg, ds = bp[offsets[0]:offsets[0] + n], bg[offsets[1]:offsets[1] + n], bs[offsets[2]:offsets[2] + n]
    dp.copy_(dev(p))
    for t in (1, 2, 3):
        gb, gf = _bf16(rng, n)
        dg.copy_(torch.from_numpy(gb.view(np.int16)).cuda().view(torch.bfloat16))
        pa.pa_adamw_step_packed_e4_bf16g(dp, dg, ds, t, **HY)
        p, st, _ = oracle.step_packed(p, gf, st, t, **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(dp), p, "p")
    assert_same_bits(host_u32(ds), st, "state")


def test_multi_bf16_gradient_list():
    import torch

    import adamw_update_gb300 as pa

    sizes = [5, 4096, 0, 30_001, 2]
    rng = np.random.default_rng(9)
    ps = [rng.normal(0, 0.02, n).astype(np.float32) for n in sizes]
    sts = [np.zeros(n, np.uint32) for n in sizes]
    dps = [dev(p) for p in ps]
    dss = [torch.zeros(n, dtype=torch.int32, device="cuda") for n in sizes]
    for t in (1, 2):
        gs = [_bf16(rng, n) for n in sizes]
        dgs = [torch.from_numpy(gb.view(np.int16)).cuda().view(torch.bfloat16) for gb, _ in gs]
        pa.pa_adamw_step_packed_e4_multi_bf16g(list(zip(dps, dgs, dss)), t, **HY)
        for k in range(len(sizes)):
            ps[k], sts[k], _ = oracle.step_packed(ps[k], gs[k][1], sts[k], t, **HY)
    torch.cuda.synchronize()
    for k in range(len(sizes)):
        assert_same_bits(host_f32(dps[k]), ps[k], f"p {k}")
        assert_same_bits(host_u32(dss[k]), sts[k], f"state {k}")


@pytest.mark.parametrize("n", [7, 6149, 20_003])
def test_one_tensor_bf16_gradient_list(n):
    """A one-tensor list of the bfloat16-gradient call (passed by value, no
    descriptor table) equals the oracle on the widened gradient."""
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(n)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = np.zeros(n, np.uint32)
    dp, ds = dev(p), torch.zeros(n, dtype=torch.int32, device="cuda")
    for t in (1, 2, 3):
        gb, gf = _bf16(rng, n)
        dg = torch.from_numpy(gb.view(np.int16)).cuda().view(torch.bfloat16)
        pa.pa_adamw_step_packed_e4_multi_bf16g([(dp, dg, ds)], t, **HY)
        p, st, _ = oracle.step_packed(p, gf, st, t, **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(dp), p, "p")
    assert_same_bits(host_u32(ds), st, "state")
