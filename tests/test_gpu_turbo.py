"""The TurboAdam-style step (pa_turbo_step) against the CPU oracle.

Each step starts the oracle from the GPU's own state before the step, so that
every step is compared from identical inputs: the parameters, the UState codes
and bf16 means, the 1Q indices and fp16 endpoints must be equal bit for bit,
and the rotated decode scale exactly.  The new encode scale comes from the RMS
accumulator, a parallel float sum on the GPU and a sequential one in the
oracle, so it is compared within the sum's rounding (the page says the same of
its own CUDA path); the accumulator itself is cleared by both.  Sizes cover
tails of storage (128) and mean (64) blocks, lanes holding 1-3 values, and
gradients that make whole blocks zero, subnormal, infinite or all equal.
"""
import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
HY = wl.HYPER
FIELDS = ("ucode", "umean", "uscal", "vidx", "vend")


def _host_state(st):
    out = {}
    for k in FIELDS:
        a = st[k].cpu().numpy()
        out[k] = a.view(np.uint16) if a.dtype == np.int16 else a.copy()
    return out


def _compare(n, p_dev, st_dev, p_exp, st_exp, what):
    got = _host_state(st_dev)
    gp = p_dev.cpu().numpy()
    nan = np.isnan(gp) & np.isnan(p_exp)
    assert np.array_equal(gp.view(np.uint32)[~nan], p_exp.view(np.uint32)[~nan]), f"{what}: p"
    for k in ("ucode", "umean", "vidx", "vend"):
        bad = np.nonzero(got[k] != st_exp[k])[0]
        assert bad.size == 0, f"{what}: {k} differs at {bad[:8]}: {got[k][bad[:8]]} vs {st_exp[k][bad[:8]]}"
    d0, e0 = got["uscal"][0], st_exp["uscal"][0]
    assert (d0 == e0 or (np.isnan(d0) and np.isnan(e0))) and got["uscal"][2] == 0.0, what
    # Two float sums of n squares, each within n * 2^-24 (relative) of the exact
    # one; the square root halves the relative difference.
    e, gv = float(st_exp["uscal"][1]), float(got["uscal"][1])
    if not (np.isnan(e) and np.isnan(gv)):  # a NaN gradient makes the tensor's RMS NaN
        tol = (n * 2.0 ** -24 + 2.0 ** -22) * abs(e)
        assert abs(gv - e) <= tol + 1e-30, (what, gv, e)


def _run(n, steps, gen, seed=0x12345678, hy=HY, factor=1.1):
    import torch

    import adamw_update_gb300 as pa

    rng = np.random.default_rng(n + 17)
    p = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).cuda()
    st = pa.turbo_state(n)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in range(1, steps + 1):
        g = gen(rng, n, t)
        before = _host_state(st)
        p_before = p.cpu().numpy()
        pa.pa_turbo_step(p, torch.from_numpy(g).cuda(), st, t, m_step_factor=factor, seed=seed,
                         nonfinite=bad, **hy)
        torch.cuda.synchronize()
        ep, est, eb = oracle.turbo_step(p_before, g, before, t, seed=seed, **hy)
        est["uscal"] = oracle.turbo_finalize(est["uscal"], n, factor)
        _compare(n, p, st, ep, est, f"n={n} step {t}")
    return int(bad.item())


def _normal(rng, n, t):
    return (rng.normal(0, 1e-3, n) * rng.choice([1.0, 10.0], n)).astype(np.float32)


@pytest.mark.parametrize("n", [1, 3, 4, 5, 63, 64, 65, 127, 128, 129, 200, 1000, 4096 + 37,
                               100_003])
def test_turbo_steps_equal_the_oracle(n):
    assert _run(n, 5, _normal) == 0


def test_turbo_large_tensor_equals_the_oracle():
    assert _run((1 << 20) + 77, 3, _normal) == 0


def test_turbo_special_blocks():
    """Blocks of zero gradients (no positive v: endpoints 0, 0), subnormal and
    huge gradients, all-equal gradients (one grid level), an infinite gradient
    (a non-finite element) and a NaN."""
    n = 128 * 8 + 40

    def gen(rng, n, t):
        g = _normal(rng, n, t)
        g[0:128] = 0.0
        g[128:256] = 1e-30 * rng.normal(size=128)
        g[256:384] = 3e4 * rng.normal(size=128)
        g[384:512] = 2e-3
        if t == 2:
            g[600] = np.inf
            g[700] = np.nan
        return g.astype(np.float32)

    assert _run(n, 4, gen) > 0


@pytest.mark.parametrize("hy", [dict(lr=1e-2, beta1=0.8, beta2=0.99, eps=1e-6, wd=0.1),
                                dict(lr=3e-4, beta1=0.95, beta2=0.9999, eps=1e-8, wd=0.0)])
def test_turbo_other_hyperparameters(hy):
    assert _run(5000, 4, _normal, seed=99, hy=hy, factor=1.3) == 0


def test_turbo_branch_free_range_edges():
    """Blocks at the edges of the ranges where the step takes the branch-free
    quotients: v' around 2^-76 at step 1 (gradients near 2^-33 on zero state),
    then |m'| just inside and just outside 2^-40 and 2^40 at step 2 (the
    gradient built from the decoded first moment, m' = b1*m + c1*g landing on
    the chosen magnitude), then an ordinary step from those states.  Blocks
    that straddle an edge take the IEEE arithmetic, the others the FMA forms;
    both must equal the oracle bit for bit."""
    import torch

    import adamw_update_gb300 as pa

    nb = 16
    n = 128 * nb
    b1, c1 = float(np.float32(HY["beta1"])), float(np.float32(1.0 - HY["beta1"]))
    rng = np.random.default_rng(404)
    p = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).cuda()
    st = pa.turbo_state(n)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    scale = rng.uniform(0.95, 1.05, n)
    sign = rng.choice([-1.0, 1.0], n)
    # per block: the step-1 gradient magnitude and the step-2 |m'| target
    # (2^-33: v' = c2*g^2 straddles 2^-76 over the block's +-5 %; 1.06 * 2^-33:
    # every v' just above it)
    g1_mag = [2.0 ** -33] * 2 + [1.06 * 2.0 ** -33] * 2 + [1e-9] * 6 + [1e-3] * 6
    m2_target = ([None] * 4 + [2.0 ** -40 * f for f in (0.5, 0.999, 1.001, 2.0, 1.0, 1.0)] +
                 [2.0 ** 40 * f for f in (0.5, 0.999, 1.001, 2.0)] + [None] * 2)
    for t in (1, 2, 3):
        before = _host_state(st)
        p_before = p.cpu().numpy()
        if t == 1:
            g = np.concatenate([sign[128 * b:128 * (b + 1)] * scale[128 * b:128 * (b + 1)] * g1_mag[b]
                                for b in range(nb)])
        elif t == 2:
            m_dec, _ = oracle.turbo_decode(before, n, 2, HY["beta1"], HY["beta2"], HY["eps"])
            g = np.empty(n)
            for b in range(nb):
                s = slice(128 * b, 128 * (b + 1))
                if m2_target[b] is None:
                    g[s] = rng.normal(0, 1e-3, 128)
                else:
                    target = sign[s] * scale[s] * m2_target[b]
                    g[s] = (target - b1 * m_dec[s].astype(np.float64)) / c1
        else:
            g = rng.normal(0, 1e-3, n)
        g = g.astype(np.float32)
        pa.pa_turbo_step(p, torch.from_numpy(g).cuda(), st, t, nonfinite=bad, **HY)
        torch.cuda.synchronize()
        ep, est, eb = oracle.turbo_step(p_before, g, before, t, **HY)
        est["uscal"] = oracle.turbo_finalize(est["uscal"], n, 1.1)
        _compare(n, p, st, ep, est, f"range edges, step {t}")
    assert int(bad.item()) == 0
