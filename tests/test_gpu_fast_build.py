"""The tolerance build (libpackedadam_fast.so, PA_FAST_MATH) against the CPU
oracle, one step from the same inputs.

That build rounds p' = p*(1-lr*wd) - upd once (one FMA) where the strict order
rounds the product and the difference separately; m', v', the divisions and
the square root are the strict ones.  So:
  * the state words (packed E4) and the blockwise codes and absmax equal the
    oracle's exactly -- stronger than the 1 code step and 1e-6 relative that
    the tolerance allows;
  * p' is within 2 ulp of the largest of |p'|, |p*dk| and |upd|: the FMA
    result differs from the strict one by at most 1/2 ulp of p*dk (the product
    the strict order rounds) plus 1/2 ulp of each of the two results.  The bound
    is in ulps of the largest term, not of p': when upd nearly cancels p*dk,
    p' is small and the two roundings of the strict order are many of its ulps
    apart from the single one;
  * the blockwise BF16 parameters are within one BF16 step.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import dev, host_f32, host_u32

pytestmark = pytest.mark.gpu
HY = wl.HYPER
PARAM_ULP_BOUND = 2.0


@pytest.fixture(scope="module")
def fast():
    import adamw_update_gb300 as pa

    return pa, pa.load_library(pa.library_path(fast=True))


def _ulp(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(np.maximum(x, np.float32(2.0 ** -126))).astype(np.float64)


def _param_error_ulps(got, p, exp):
    """|got - exp| in ulps of the largest of |exp|, |p*dk| and |exp - p*dk|."""
    pd = p * np.float32(1 - HY["lr"] * HY["wd"])
    upd = pd.astype(np.float64) - exp.astype(np.float64)
    scale = np.maximum(np.maximum(np.abs(exp), np.abs(pd)), np.abs(upd).astype(np.float32))
    return np.abs(got.astype(np.float64) - exp.astype(np.float64)) / _ulp(scale)


def _inputs(rng, n):
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = (1e-3 * rng.standard_t(3, n)).astype(np.float32)
    # near-cancelling cases: an update about as large as the decayed parameter
    k = n // 8
    p[:k] = (np.sign(g[:k]) * rng.uniform(5e-4, 2e-3, k)).astype(np.float32)
    st, _ = oracle.encode_state(rng.normal(0, 1e-3, n), np.abs(rng.normal(0, 1e-3, n)))
    return p, g, st


@pytest.mark.parametrize("step", [1, 7, 100_000])
def test_fast_build_packed_e4_within_tolerance(fast, step):
    import torch

    pa, lib = fast
    n = (1 << 20) + 3
    p, g, st = _inputs(np.random.default_rng(1), n)
    dp, ds = dev(p), dev(st)
    rc = lib.pa_adamw_step_packed_e4(dp.data_ptr(), dev(g).data_ptr(), ds.data_ptr(), n, step,
                                     HY["lr"], HY["beta1"], HY["beta2"], HY["eps"], HY["wd"],
                                     None, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ep, ew, _ = oracle.step_packed(p, g, st, step, **HY)
    gp, gw = host_f32(dp), host_u32(ds)
    assert np.array_equal(gw, ew), f"step {step}: state words differ"
    err = _param_error_ulps(gp, p, ep)
    assert err.max() <= PARAM_ULP_BOUND, f"step {step}: params {err.max():.2f} ulp"


def test_fast_build_fp32_mode_within_tolerance(fast):
    import torch

    pa, lib = fast
    n = (1 << 20) + 1
    rng = np.random.default_rng(3)
    p, g, _ = _inputs(rng, n)
    m = rng.normal(0, 1e-3, n).astype(np.float32)
    v = np.abs(rng.normal(0, 1e-6, n)).astype(np.float32)
    dp, dm, dv = dev(p), dev(m), dev(v)
    rc = lib.pa_adamw_step_fp32(dp.data_ptr(), dev(g).data_ptr(), dm.data_ptr(), dv.data_ptr(), n,
                                5, HY["lr"], HY["beta1"], HY["beta2"], HY["eps"], HY["wd"], None,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ep, em, ev, _ = oracle.step_fp32(p, g, m, v, 5, **HY)
    assert np.array_equal(host_f32(dm).view(np.uint32), em.view(np.uint32))
    assert np.array_equal(host_f32(dv).view(np.uint32), ev.view(np.uint32))
    err = _param_error_ulps(host_f32(dp), p, ep)
    assert err.max() <= PARAM_ULP_BOUND, f"params {err.max():.2f} ulp"


def test_fast_build_blockwise_within_tolerance(fast):
    import torch

    pa, lib = fast
    n = 64 * 2048 + 100
    nb = -(-n // 2048)
    rng = np.random.default_rng(2)
    q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    mc = rng.integers(0, 256, n).astype(np.uint8)
    vc = rng.integers(0, 256, n).astype(np.uint8)
    ma = np.abs(rng.normal(0, 1e-3, nb)).astype(np.float32)
    va = np.abs(rng.normal(0, 1e-6, nb)).astype(np.float32)
    d = [dev(x) for x in (p, g)] + [torch.empty(n, dtype=torch.bfloat16, device="cuda")]
    d += [dev(mc), dev(ma), dev(vc), dev(va), dev(q1), dev(q2)]
    rc = lib.pa_adamw_step_blockwise8(*[t.data_ptr() for t in d], n, 3, HY["lr"], HY["beta1"],
                                      HY["beta2"], HY["eps"], HY["wd"], None,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ob, emc, ema, evc, eva, _ = oracle.step_blockwise8(p, g, mc, ma, vc, va, q1, q2, 3, **HY)
    gb = d[2].view(torch.int16).cpu().numpy().view(np.uint16).astype(np.int64)
    assert np.abs(gb - ob.astype(np.int64)).max() <= 1  # BF16 within one step
    assert np.array_equal(host_f32(d[4]).view(np.uint32), ema.view(np.uint32))
    assert np.array_equal(host_f32(d[6]).view(np.uint32), eva.view(np.uint32))
    assert np.array_equal(d[3].cpu().numpy(), emc)
    assert np.array_equal(d[5].cpu().numpy(), evc)
