"""GPU 8-bit blockwise step against the CPU oracle, bit for bit, through the C
ABI (KBench "quantized-optimizer-state" reference.py, quantized_adamw_step and
_requantise): BF16 parameters, both code arrays and both absmax arrays, over
several steps with p fed back as fp32(p_bf16), on whole and short last blocks
and on several ascending maps."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_same_f32_nan_aware, dev, host_f32

pytestmark = pytest.mark.gpu

HY = wl.HYPER


@pytest.fixture(scope="module")
def pa():
    import adamw_update_gb300

    return adamw_update_gb300


def _maps(kind):
    if kind == "dynamic":
        return wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
    if kind == "linear":
        return wl.linear_qmap_signed(), wl.linear_qmap_unsigned()
    return wl.random_qmap(1, True), wl.random_qmap(2, False)


def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _run(pa, n, kind, steps=3, g_scale=1e-3, inject=None, seed=0):
    import torch

    q1, q2 = _maps(kind)
    nb = -(-n // 2048)
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    mc = np.full(n, wl.nearest_zero_code(q1), np.uint8)
    vc = np.full(n, wl.nearest_zero_code(q2), np.uint8)
    ma = np.zeros(nb, np.float32)
    va = np.zeros(nb, np.float32)
    d_mc, d_vc, d_ma, d_va = dev(mc), dev(vc), dev(ma), dev(va)
    d_q1, d_q2 = dev(q1), dev(q2)
    d_out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    e_bad = 0
    for t in range(1, steps + 1):
        g = rng.normal(0, g_scale, n).astype(np.float32)
        if inject is not None and t == 2:
            g[inject] = np.nan
        pa.pa_adamw_step_blockwise8(dev(p), dev(g), d_out, d_mc, d_ma, d_vc, d_va, d_q1, d_q2,
                                    t, nonfinite=bad, **HY)
        ob, mc, ma, vc, va, b = oracle.step_blockwise8(p, g, mc, ma, vc, va, q1, q2, t, **HY)
        e_bad += b
        torch.cuda.synchronize()
        got = d_out.view(torch.int16).cpu().numpy().view(np.uint16)
        nan = np.isnan(_bf16_to_f32(ob))
        assert np.array_equal(np.isnan(_bf16_to_f32(got)), nan)
        assert np.array_equal(got[~nan], ob[~nan]), f"bf16 p, step {t}"
        assert np.array_equal(d_mc.cpu().numpy(), mc), f"m codes, step {t}"
        assert np.array_equal(d_vc.cpu().numpy(), vc), f"v codes, step {t}"
        assert_same_f32_nan_aware(host_f32(d_ma), ma, f"m absmax, step {t}")
        assert_same_f32_nan_aware(host_f32(d_va), va, f"v absmax, step {t}")
        p = _bf16_to_f32(ob)  # the next step reads the widened BF16 output
    assert int(bad.item()) == e_bad


@pytest.mark.parametrize("n", [1, 5, 2048, 2049, 3 * 2048 + 777, 40 * 2048])
def test_blockwise_sizes(pa, n):
    _run(pa, n, "dynamic")


@pytest.mark.parametrize("kind", ["linear", "random"])
def test_blockwise_maps(pa, kind):
    _run(pa, 5 * 2048 + 100, kind, seed=4)


def test_blockwise_large_gradients_and_nan(pa):
    """A NaN makes its block's absmax NaN and is counted; other blocks are
    unaffected."""
    _run(pa, 6 * 2048 + 3, "dynamic", g_scale=10.0, inject=[5, 4097], seed=8)


def test_blockwise_alignment_errors(pa):
    import torch

    x = torch.zeros(4096 + 8, dtype=torch.float32, device="cuda")
    b = torch.zeros(4096 + 8, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(4096 + 8, dtype=torch.uint8, device="cuda")
    q = dev(wl.dynamic_qmap_signed())
    with pytest.raises(pa.PackedAdamError):
        pa.pa_adamw_step_blockwise8(x[1:4097], x[:4096], b[:4096], c[:4096], x[:2], c[:4096],
                                    x[:2], q, q, 1)


def test_blockwise_tensor_list_equals_single_calls(pa):
    """One launch over a list (short, whole and ragged tensors, an empty one)
    gives the bits of one single-tensor call per tensor, and of the oracle."""
    import torch

    q1, q2 = _maps("dynamic")
    sizes = [1, 2048, 2049, 0, 5000, 3 * 2048 + 7]
    rng = np.random.default_rng(12)
    lists, singles, host = [], [], []
    for n in sizes:
        nb = -(-n // 2048)
        p = rng.normal(0, 0.02, n).astype(np.float32)
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        mc = np.full(n, wl.nearest_zero_code(q1), np.uint8)
        vc = np.full(n, wl.nearest_zero_code(q2), np.uint8)
        z = np.zeros(nb, np.float32)
        mk = lambda: (dev(p), dev(g), torch.empty(n, dtype=torch.bfloat16, device="cuda"),  # noqa: E731
                      dev(mc), dev(z), dev(vc), dev(z))
        lists.append(mk())
        singles.append(mk())
        host.append([p, g, mc, z.copy(), vc, z.copy()])
    d1, d2 = dev(q1), dev(q2)
    for t in (1, 2):
        pa.pa_adamw_step_blockwise8_multi(lists, d1, d2, t, **HY)
        for e in singles:
            if e[0].numel():
                pa.pa_adamw_step_blockwise8(*e, d1, d2, t, **HY)
        torch.cuda.synchronize()
        for k, (a, b) in enumerate(zip(lists, singles)):
            for x, y in zip(a[2:], b[2:]):
                xb = x.cpu().numpy().view(np.uint8) if x.dtype != torch.bfloat16 else \
                    x.view(torch.int16).cpu().numpy().view(np.uint8)
                yb = y.cpu().numpy().view(np.uint8) if y.dtype != torch.bfloat16 else \
                    y.view(torch.int16).cpu().numpy().view(np.uint8)
                assert np.array_equal(xb, yb), (k, t)
            if sizes[k]:
                p, g, mc, ma, vc, va = host[k]
                ob, mc, ma, vc, va, _ = oracle.step_blockwise8(p, g, mc, ma, vc, va, q1, q2, t, **HY)
                host[k] = [p, g, mc, ma, vc, va]
                got = a[2].view(torch.int16).cpu().numpy().view(np.uint16)
                assert np.array_equal(got, ob) and np.array_equal(a[3].cpu().numpy(), mc)
                assert np.array_equal(a[5].cpu().numpy(), vc)
