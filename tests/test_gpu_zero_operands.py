"""Zero and tiny operands of the division and square roots, bit for bit
against the CPU oracle.

The step kernels keep exactly-zero gradients on zero state off the slow path
of CUDA's correctly rounded division and square root: a warp holding such a
gradient divides v' by bc2 with Markstein's method (rb = RN(1/bc2)), takes
u/den with u = +-0 as u, and the roots of a zero v'/bc2 or v' as that zero.
These tests feed what those substitutions must leave untouched: +-0 and
subnormal gradients, gradients whose square underflows, zero and random prior
state (every E4 code; binary16 words with NaN and Inf codes), p = +-0, and
hyperparameters at the edges (eps = 0, where den may be 0; eps far below the
root of the smallest normal; bc2 near 0, outside the Markstein range; lr = 0;
early and late steps, where bc2 rounds to 1).
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_same_bits, assert_same_f32_nan_aware, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu

HYPERS = [
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01),
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=0.0, wd=0.01),     # no floor: den may be 0
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-30, wd=0.0),    # eps below the floor's root
    dict(lr=2e-2, beta1=0.5, beta2=1.0 - 1e-9, eps=1e-8, wd=0.1),  # bc2 ~ 1e-9: no floor
    dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-3, wd=0.0),      # u == 0 everywhere
]
STEPS = [1, 40_000]  # an early step and one where 1 - beta2^step rounds to 1


@pytest.fixture(scope="module")
def pa():
    import adamw_update_gb300

    return adamw_update_gb300


def _gradients(rng, n):
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    kind = rng.integers(0, 20, n)
    g[kind < 5] = 0.0                                            # +0
    g[kind == 5] = -0.0                                          # -0
    sub = kind == 6                                              # subnormal
    g[sub] = (rng.integers(1, 1 << 23, sub.sum()).astype(np.uint32)
              | (rng.integers(0, 2, sub.sum()).astype(np.uint32) << 31)).view(np.float32)
    tiny = kind == 7                                             # g*g underflows
    g[tiny] = (10.0 ** rng.uniform(-37, -20, tiny.sum()) * rng.choice([-1, 1], tiny.sum())
               ).astype(np.float32)
    return g


def _params(rng, n):
    p = rng.normal(0, 0.02, n).astype(np.float32)
    p[::97] = 0.0
    p[1::97] = -0.0
    return p


def _state(rng, n):
    s = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    s[rng.random(n) < 0.5] = 0  # zero state: the fresh-zero case
    s[::13] = 0x8000  # m = -0, RMS 0
    return s


@pytest.mark.parametrize("mode", ["e4", "fp16"])
@pytest.mark.parametrize("step", STEPS)
@pytest.mark.parametrize("hy", HYPERS)
def test_packed_zero_operands(pa, mode, step, hy):
    import torch

    n = 3 * 16384 + 4097  # several chunks and a ragged tail
    rng = np.random.default_rng(step + 7 * len(mode) + int(hy["eps"] > 0))
    p, st = _params(rng, n), _state(rng, n)
    gs = [_gradients(rng, n) for _ in range(2)]
    dp, ds = dev(p), dev(st)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = pa.pa_adamw_step_packed_e4 if mode == "e4" else pa.pa_adamw_step_packed_fp16
    eb = 0
    for k, g in enumerate(gs):
        fn(dp, dev(g), ds, step + k, nonfinite=bad, **hy)
        p, st, b = oracle.step_packed(p, g, st, step + k, mode=mode, **hy)
        eb += b
    torch.cuda.synchronize()
    assert_same_f32_nan_aware(host_f32(dp), p, f"{mode} p")
    assert_same_bits(host_u32(ds), st, f"{mode} state")
    assert int(bad.item()) == eb


@pytest.mark.parametrize("step", STEPS)
@pytest.mark.parametrize("hy", HYPERS)
def test_fp32_zero_operands(pa, step, hy):
    """FP32 moments read from memory may be zero, -0, subnormal, negative,
    NaN or Inf; the multi-tensor path (16-byte and 4-byte accesses)."""
    import torch

    n = 2 * 16384 + 333
    rng = np.random.default_rng(step + 3)
    p = _params(rng, n)
    m = rng.normal(0, 1e-4, n).astype(np.float32)
    v = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
    zero = rng.random(n) < 0.4
    m[zero] = 0.0
    v[zero] = 0.0
    v[5::101] = -1e-6
    v[6::101] = np.nan
    v[7::101] = np.inf
    v[8::101] = np.float32(1e-40)
    m[9::101] = -0.0
    g = _gradients(rng, n)
    dp, dm, dv = dev(p), dev(m), dev(v)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    pa.pa_adamw_step_fp32(dp, dev(g), dm, dv, step, nonfinite=bad, **hy)
    ep, em, ev, eb = oracle.step_fp32(p, g, m, v, step, **hy)
    torch.cuda.synchronize()
    assert_same_f32_nan_aware(host_f32(dp), ep, "p")
    assert_same_f32_nan_aware(host_f32(dm), em, "m")
    assert_same_f32_nan_aware(host_f32(dv), ev, "v")
    assert int(bad.item()) == eb
