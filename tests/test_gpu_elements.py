"""The update element on adversarial inputs, GPU against the CPU oracle, bit
for bit: exact zeros of either sign, subnormals, magnitudes from 1e-12 to 10,
second moments down to 1e-30, first moments that nearly cancel the new
gradient term, updates about as large as the decayed parameter -- at early
steps and at steps where 1 - beta2**step rounds to 1.  The FP32 mode takes m
and v as given, so every path of the element is reached (plain and zero-safe
warps, UNIT_BC2); the packed modes take the same p and g with random state
words."""
import numpy as np
import pytest

import oracle
import pins
from gpu_helpers import assert_same_bits, assert_same_f32_nan_aware, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu
N = 200_003


@pytest.mark.parametrize("step", [1, 10, 20_000])
@pytest.mark.parametrize("hy", pins.HYPER_SETS, ids=["default", "large_lr", "no_wd"])
def test_fp32_mode_adversarial_elements(step, hy):
    import torch

    import adamw_update_gb300 as pa

    p, g, m, v = pins._adversarial_elements(np.random.default_rng(step), N)
    dp, dm, dv = dev(p), dev(m), dev(v)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    pa.pa_adamw_step_fp32(dp, dev(g), dm, dv, step, nonfinite=bad, **hy)
    torch.cuda.synchronize()
    ep, em, ev, eb = oracle.step_fp32(p, g, m, v, step, **hy)
    assert_same_f32_nan_aware(host_f32(dp), ep, "p'")
    assert_same_f32_nan_aware(host_f32(dm), em, "m'")
    assert_same_f32_nan_aware(host_f32(dv), ev, "v'")
    assert int(bad.item()) == eb


@pytest.mark.parametrize("mode", ["e4", "fp16"])
@pytest.mark.parametrize("step", [1, 20_000])
def test_packed_modes_adversarial_elements(mode, step):
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(100 + step)
    p, g, _, _ = pins._adversarial_elements(rng, N)
    w = pins._random_state_words(rng, N, mode)
    dp, dw = dev(p), dev(w)
    fn = pa.pa_adamw_step_packed_e4 if mode == "e4" else pa.pa_adamw_step_packed_fp16
    hy = pins.HYPER_SETS[0]
    fn(dp, dev(g), dw, step, **hy)
    torch.cuda.synchronize()
    ep, ew, _ = oracle.step_packed(p, g, w, step, mode=mode, **hy)
    assert_same_f32_nan_aware(host_f32(dp), ep, "p'")
    assert_same_bits(host_u32(dw), ew, "state words")
