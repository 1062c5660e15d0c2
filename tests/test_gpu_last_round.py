"""Staged steps over more tiles than one round of CTAs (grid = one CTA per
SM, 152 on GB300), whose last round is partial and holds the ragged ends of
the list: a tensor's head peel (its views start off a 16-byte boundary), a
short last tile with a ragged tail of fewer than one staging unit, a tensor
on the 4-byte path (mismatched offsets) and a 3-element tensor.  Every case
is bit for bit equal to the oracle ("Packed AdamW / Reference / v1.0.0",
"Release scope"; the FP16 and FP32 comparison modes of the "Packed AdamW
Reference" README).

Sizes (6144 elements per tile):
  156 * 6144 + 1234  157 tiles: five in the last round, the last one short
  212 * 6144 + 10    213 tiles: 61 in the last round (the gpt-52 list has
                     1575 tiles, 55 in its last round)
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_same_bits, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu
HY = wl.HYPER
TILE = 6144
SIZES = [156 * TILE + 1234, 212 * TILE + 10]


def _views(n, offsets, dtypes):
    import torch

    return [torch.zeros(n + 8, dtype=dt, device="cuda")[o:o + n] for o, dt in zip(offsets, dtypes)]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("mode,offsets", [("e4", (0, 0, 0)), ("e4", (1, 1, 1)),
                                          ("e4", (1, 2, 3)), ("fp16", (3, 3, 3)),
                                          ("fp32", (2, 2, 2, 2))])
def test_single_tensor(n, mode, offsets):
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(n + sum(offsets))
    p = rng.normal(0, 0.02, n).astype(np.float32)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    if mode == "fp32":
        dp, dg, dm, dv = _views(n, offsets, [torch.float32] * 4)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
    else:
        dp, dg, ds = _views(n, offsets, [torch.float32, torch.float32, torch.int32])
        st = np.zeros(n, np.uint32)
    dp.copy_(dev(p))
    for t in (1, 2):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        dg.copy_(dev(g))
        if mode == "fp32":
            pa.pa_adamw_step_fp32(dp, dg, dm, dv, t, nonfinite=bad, **HY)
            p, m, v, _ = oracle.step_fp32(p, g, m, v, t, **HY)
        else:
            fn = pa.pa_adamw_step_packed_e4 if mode == "e4" else pa.pa_adamw_step_packed_fp16
            fn(dp, dg, ds, t, nonfinite=bad, **HY)
            p, st, _ = oracle.step_packed(p, g, st, t, mode=mode, **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(dp), p, f"{mode} p")
    if mode == "fp32":
        assert_same_bits(host_f32(dm), m, "m")
        assert_same_bits(host_f32(dv), v, "v")
    else:
        assert_same_bits(host_u32(ds), st, f"{mode} state")
    assert int(bad.item()) == 0


@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 5, 1)])
def test_single_tensor_bf16_gradients(offsets):
    import torch

    import adamw_update_gb300 as pa

    n = SIZES[0]
    rng = np.random.default_rng(7 + sum(offsets))
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = np.zeros(n, np.uint32)
    dp, dg, ds = _views(n, offsets, [torch.float32, torch.bfloat16, torch.int32])
    dp.copy_(dev(p))
    for t in (1, 2):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        bits = (g.view(np.uint32) >> 16).astype(np.uint16)
        dg.copy_(torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16))
        pa.pa_adamw_step_packed_e4_bf16g(dp, dg, ds, t, **HY)
        p, st, _ = oracle.step_packed(p, (bits.astype(np.uint32) << 16).view(np.float32), st, t,
                                      **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(dp), p, "p")
    assert_same_bits(host_u32(ds), st, "state")


# 157 tiles: the last round holds tiles 1 and 2 of tensor 1, tensor 2 whole
# (a head peel: its views start one element in), tensor 3 (mismatched
# offsets: the 4-byte path) and the 3-element tensor 4.
LIST = [(150 * TILE + 100, 0, 0, 0), (2 * TILE + 5, 0, 0, 0), (4100, 1, 1, 1),
        (5000, 1, 2, 3), (3, 2, 2, 2)]


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_list(mode):
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(11)
    host, views = [], []
    for n, *off in LIST:
        p = rng.normal(0, 0.02, n).astype(np.float32)
        if mode == "fp32":
            v = _views(n, off + [off[-1]], [torch.float32] * 4)
            host.append([p, np.zeros(n, np.float32), np.zeros(n, np.float32)])
        else:
            v = _views(n, off, [torch.float32, torch.float32, torch.int32])
            host.append([p, np.zeros(n, np.uint32)])
        v[0].copy_(dev(p))
        views.append(v)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = {"e4": pa.pa_adamw_step_packed_e4_multi, "fp16": pa.pa_adamw_step_packed_fp16_multi,
          "fp32": pa.pa_adamw_step_fp32_multi}[mode]
    for t in (1, 2):
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n, *_ in LIST]
        for v, g in zip(views, gs):
            v[1].copy_(dev(g))
        fn([tuple(v) for v in views], t, nonfinite=bad, **HY)
        for h, g in zip(host, gs):
            if mode == "fp32":
                h[0], h[1], h[2], _ = oracle.step_fp32(h[0], g, h[1], h[2], t, **HY)
            else:
                h[0], h[1], _ = oracle.step_packed(h[0], g, h[1], t, mode=mode, **HY)
    torch.cuda.synchronize()
    for k, (h, v) in enumerate(zip(host, views)):
        assert_same_bits(host_f32(v[0]), h[0], f"tensor {k} p")
        for a, d in zip(h[1:], v[2:]):
            got = host_u32(d) if a.dtype == np.uint32 else host_f32(d)
            assert_same_bits(got, a, f"tensor {k} state")
    assert int(bad.item()) == 0


def test_graph_step_list():
    """The graph-replayable step over the same list (uncaptured calls)."""
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(12)
    host, views = [], []
    for n, *off in LIST:
        p = rng.normal(0, 0.02, n).astype(np.float32)
        v = _views(n, off, [torch.float32, torch.float32, torch.int32])
        v[0].copy_(dev(p))
        host.append([p, np.zeros(n, np.uint32)])
        views.append(v)
    rows = torch.empty(4 * 8, dtype=torch.float32, device="cuda")
    pa.pa_hyper_table_fill(rows, 1, 4, **HY)
    index = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in (1, 2):
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n, *_ in LIST]
        for v, g in zip(views, gs):
            v[1].copy_(dev(g))
        pa.pa_adamw_step_packed_e4_multi_graph([tuple(v) for v in views], rows, 4, index)
        for h, g in zip(host, gs):
            h[0], h[1], _ = oracle.step_packed(h[0], g, h[1], t, **HY)
    torch.cuda.synchronize()
    for k, (h, v) in enumerate(zip(host, views)):
        assert_same_bits(host_f32(v[0]), h[0], f"tensor {k} p")
        assert_same_bits(host_u32(v[2]), h[1], f"tensor {k} state")
