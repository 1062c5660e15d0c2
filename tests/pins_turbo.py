"""Pins for the TurboAdam-style oracle (oracle/turbo.c): each check compares it
with something other than itself -- closed forms of the grid, numpy's binary16
conversion, the FP32 AdamW step of oracle.c on the decoded moments (itself
pinned in pins.py), unbiasedness of both stochastic roundings, the page's
reconstruction identity, the mean preservation of the recentring, and
statistical properties of the counter hash.

"TurboAdam" README (turboadam 0.2.0), "How it works": "UState: first-moment
compression", "1Q: second-moment compression", "The AdamW update remains
AdamW", "Fused CUDA path"; the readings T1-T9 are in turbo.c's header.

Every ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch; test_turbo_oracle.py runs them on the oracle and on planted mistakes.
"""
from __future__ import annotations

import numpy as np

import oracle as _oracle_mod
from pins import assert_bits_equal

HY = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
K = 15  # 4-bit 1Q: indices 1..15 are grid levels


# ---- the counter hash (T3) ---------------------------------------------------

def check_uniform_statistics(orc):
    """u in [0, 1) on the 2^-24 grid; mean, 64-bin histogram and lag-1
    correlation of 2^20 values per stream as for i.i.d. uniforms; different
    streams, steps and seeds give unrelated sequences."""
    n = 1 << 20
    idx = np.arange(n, dtype=np.uint64)
    seqs = {}
    for key in ((7, 1, 1), (7, 1, 2), (7, 2, 1), (8, 1, 1)):
        u = orc.turbo_uniform(key[0], key[1], key[2], idx).astype(np.float64)
        assert u.min() >= 0.0 and u.max() < 1.0
        assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
        assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n), key
        h = np.bincount((u * 64).astype(int), minlength=64)
        chi2 = float(((h - n / 64) ** 2 / (n / 64)).sum())
        assert chi2 < 130.0, (key, chi2)  # df 63: P(chi2 > 130) ~ 1e-6
        c = np.corrcoef(u[:-1], u[1:])[0, 1]
        assert abs(c) < 6 / np.sqrt(n), (key, c)
        seqs[key] = u
    keys = list(seqs)
    for a in range(len(keys)):
        for b in range(a + 1, len(keys)):
            c = np.corrcoef(seqs[keys[a]], seqs[keys[b]])[0, 1]
            assert abs(c) < 6 / np.sqrt(n), (keys[a], keys[b], c)


def check_two_uniforms_per_output(orc):
    """Indices 2k and 2k+1 of a stream take bits 40..63 and 16..39 of the one
    SplitMix64 output at counter (step, stream, k): both on the 2^-24 grid,
    and together they are 48 bits of that output."""
    rng = np.random.default_rng(9)
    for _ in range(300):
        seed = int(rng.integers(0, 2 ** 63))
        step, stream, k = int(rng.integers(1, 2 ** 20)), int(rng.integers(1, 3)), int(rng.integers(0, 2 ** 38))
        c = (step << 42) | (stream << 40) | k
        h = orc.splitmix64_at(seed, c)
        u = orc.turbo_uniform(seed, step, stream, np.array([2 * k, 2 * k + 1], np.uint64))
        assert int(np.float64(u[0]) * 2 ** 24) == h >> 40
        assert int(np.float64(u[1]) * 2 ** 24) == (h >> 16) & 0xFFFFFF


def check_counter_is_a_splitmix_position(orc):
    """Counter c of seed s is output number c+1 of the generator whose state
    starts at s and advances by the golden-ratio increment: moving one step
    along the counter equals moving the seed by one increment; and the mixing
    function avalanches (each input bit flips each output bit about half the
    time)."""
    gamma = 0x9E3779B97F4A7C15
    rng = np.random.default_rng(5)
    for _ in range(200):
        seed = int(rng.integers(0, 2 ** 63))
        c = int(rng.integers(1, 2 ** 40))
        assert orc.splitmix64_at(seed, c) == orc.splitmix64_at((seed + gamma) % 2 ** 64, c - 1)
    flips = np.zeros(64)
    trials = 400
    for t in range(trials):
        x = int(rng.integers(0, 2 ** 63))
        base = orc.splitmix64_at(x, 0)
        for bit in range(64):
            flips[bit] += bin(base ^ orc.splitmix64_at(x ^ (1 << bit), 0)).count("1")
    mean_flips = flips / trials
    assert np.all(np.abs(mean_flips - 32) < 3), mean_flips


# ---- 1Q (T1, T2) ---------------------------------------------------------------

def check_q1_grid_closed_forms(orc):
    """Level 0 is 0; level 1 is 2^lo and level 15 is 2^hi; across 14 binades
    the grid is exactly the powers of two; within one binade it is linear in
    value; it is strictly increasing."""
    for lo in (-126, -40, -20, 0, 100, 113):
        lv = orc.q1_levels(lo, lo + 14)
        assert lv[0] == 0.0
        assert_bits_equal(lv[1:], np.ldexp(1.0, np.arange(lo, lo + 15)), f"powers from {lo}")
    # below 2^-126 the bit pattern is linear in value: 2^-149 .. 2^-135 evenly
    lv = orc.q1_levels(-149, -135).astype(np.float64)
    assert lv[1] == 2.0 ** -149 and lv[15] == 2.0 ** -135
    assert np.all(np.abs(np.diff(lv[1:]) - (2.0 ** -135 - 2.0 ** -149) / 14) <= 2.0 ** -149)
    for lo in (-126, -30, -3, 60):
        lv = orc.q1_levels(lo, lo + 1).astype(np.float64)
        step = 2.0 ** lo / 14
        assert np.all(np.abs(np.diff(lv[1:]) - step) <= 2.0 ** (lo - 23) * 1.01), lo
    for lo, hi in ((-140, -120), (-60, -2), (-20, -10), (3, 4), (-1, 126)):
        lv = orc.q1_levels(lo, hi)
        assert lv[1] == 2.0 ** lo and lv[15] == np.float32(2.0 ** hi)
        assert np.all(np.diff(lv) > 0), (lo, hi)
    assert np.all(orc.q1_levels(-7, -7)[1:] == 2.0 ** -7)


def check_q1_endpoints(orc):
    """The endpoints are the binary exponents bracketing the block's positive
    values (2^lo <= smallest < 2^(lo+1), 2^(hi-1) < largest <= 2^hi); zeros,
    NaN and Inf do not count; no positive value gives (0, 0); the fp16 codes of
    the integer endpoints are numpy's binary16 of them, for every exponent."""
    rng = np.random.default_rng(9)
    for trial in range(300):
        cnt = int(rng.integers(1, 129))
        v = (10.0 ** rng.uniform(-44, 38, cnt) * (rng.random(cnt) < 0.9)).astype(np.float32)
        if trial % 7 == 0:
            v[0] = np.nan
        if trial % 11 == 0:
            v[-1] = np.inf
        lo, hi = orc.q1_endpoints(v)
        pos = v[np.isfinite(v) & (v > 0)].astype(np.float64)
        if pos.size == 0:
            assert (lo, hi) == (0, 0)
            continue
        mn, mx = pos.min(), pos.max()
        assert 2.0 ** lo <= mn < 2.0 ** (lo + 1), (mn, lo)
        assert mx <= 2.0 ** hi and (hi == 127 or 2.0 ** (hi - 1) < mx), (mx, hi)
    assert orc.q1_endpoints(np.zeros(5, np.float32)) == (0, 0)
    for e in range(-149, 128):
        h = orc.q1_endpoint_code(e)
        assert h == int(np.float16(e).view(np.uint16)), e
        assert orc.q1_endpoint_value(h) == e


def check_q1_rounding(orc):
    """Zero goes to index 0 and a grid value to its own index whatever u; any
    other value to one of the two levels around it, the upper one exactly
    when u lies below the value's fraction of the gap, so that over a uniform
    grid of u the mean decoded value is the value itself."""
    rng = np.random.default_rng(10)
    lo, hi = -24, -9
    lv = orc.q1_levels(lo, hi).astype(np.float64)
    us = ((np.arange(1024) + 0.5) / 1024).astype(np.float32)
    for k in range(16):
        assert np.all(orc.q1_index(np.full(4, lv[k], np.float32), lo, hi, us[::256]) == k)
    v = (2.0 ** rng.uniform(lo, hi, 300)).astype(np.float32)
    for x in v:
        idx = orc.q1_index(np.full(us.size, x, np.float32), lo, hi, us)
        d = lv[idx]
        j = np.searchsorted(lv, float(x), side="right") - 1
        assert set(np.unique(idx)) <= {j, j + 1}
        assert np.all(np.diff(idx) <= 0)  # larger u never rounds up more
        gap = lv[min(j + 1, 15)] - lv[j]
        assert abs(d.mean() - float(x)) <= gap / 1024 + 1e-7 * float(x), (x, d.mean())


# ---- UState (T4) ------------------------------------------------------------------

def check_ustate_code(orc):
    """Inside [-1.5 s, 1.5 s] a residual rounds to one of the two levels around
    it, unbiased over a uniform grid of u; beyond, it saturates at the end
    levels; with s = 0 every residual is the zero-mean pair of middle levels."""
    lv = np.array([-1.5, -0.5, 0.5, 1.5])
    us = ((np.arange(512) + 0.5) / 512).astype(np.float32)
    rng = np.random.default_rng(11)
    for s in (1e-3, 0.7, 3.0):
        for r in rng.uniform(-1.5 * s, 1.5 * s, 200).astype(np.float32):
            c = orc.ustate_code(np.full(us.size, r, np.float32), s, us)
            assert np.ptp(c) <= 1
            got = (lv[c] * s).mean()
            assert abs(got - float(r)) <= s / 512 + 1e-6 * s, (s, r, got)
        big = np.float32(1.5 * s * 1.01)
        assert np.all(orc.ustate_code(np.full(8, big, np.float32), s, us[::64]) == 3)
        assert np.all(orc.ustate_code(np.full(8, -big, np.float32), s, us[::64]) == 0)
    c = orc.ustate_code(np.full(us.size, 0.37, np.float32), 0.0, us)
    assert set(np.unique(c)) == {1, 2} and abs(lv[c].mean()) < 1e-9


# ---- the step -------------------------------------------------------------------------

def _run(orc, n, steps, seed=0x12345678, gscale=1e-3, gen=1):
    rng = np.random.default_rng(gen)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = _oracle_mod.turbo_zero_state(n)
    hist = []
    for t in range(1, steps + 1):
        g = (rng.normal(0, gscale, n) * rng.choice([1.0, 10.0], n)).astype(np.float32)
        hist.append((t, p.copy(), g, {k: v.copy() for k, v in st.items()}))
        p, st, bad = orc.turbo_step(p, g, st, t, seed=seed, **HY)
        assert bad == 0
        st["uscal"] = orc.turbo_finalize(st["uscal"], n)
    return p, st, hist


def check_step_is_adamw_on_decoded_moments(orc):
    """At every step the parameter is, bit for bit, the FP32 AdamW step (oracle.c)
    from the prior moments that the state decodes to; at step 1 from zero
    state these are m = v = 0."""
    n = 1000 + 37
    _, _, hist = _run(orc, n, 6)
    for t, p, g, st in hist:
        m, v = orc.turbo_decode(st, n, t, HY["beta1"], HY["beta2"], HY["eps"])
        if t == 1:
            assert not m.any() and not v.any()
        p1, _, _ = orc.turbo_step(p, g, st, t, **HY)
        pf, mf, vf, _ = orc.step_fp32(p, g, m, v, t, **HY)
        assert_bits_equal(p1, pf, f"p' at step {t}")


def check_second_moment_bracketed_and_unbiased(orc):
    """The persisted second moment decodes to one of the two grid levels around
    the exact v' of the step (the grid of its block's new endpoints), and its
    mean over many seeds is v'."""
    n = 512
    _, _, hist = _run(orc, n, 3)
    t, p, g, st = hist[-1]
    m, v = orc.turbo_decode(st, n, t, HY["beta1"], HY["beta2"], HY["eps"])
    _, _, vexact, _ = orc.step_fp32(p, g, m, v, t, **HY)
    acc = np.zeros(n)
    seeds = 200
    for s in range(seeds):
        _, st1, _ = orc.turbo_step(p, g, st, t, seed=1000 + s, **HY)
        _, vhat = orc.turbo_decode(st1, n, t + 1, HY["beta1"], HY["beta2"], HY["eps"])
        for b in range(n // 128):
            sl = slice(128 * b, 128 * b + 128)
            lo = orc.q1_endpoint_value(int(st1["vend"][2 * b]))
            hi = orc.q1_endpoint_value(int(st1["vend"][2 * b + 1]))
            lv = orc.q1_levels(lo, hi).astype(np.float64)
            j = np.searchsorted(lv, vexact[sl].astype(np.float64), side="right") - 1
            ok = (vhat[sl] == lv[j]) | (vhat[sl] == lv[np.minimum(j + 1, 15)])
            assert ok.all(), (s, b)
        acc += vhat
    rel = (acc / seeds - vexact) / vexact
    assert abs(rel.mean()) < 3e-3, rel.mean()


def check_first_moment_reconstructed(orc):
    """"An unquantized q_t reconstructs m_t exactly" given the persisted second
    moment: the UState code rounds q_t without bias, so over many seeds the
    first moment the next step decodes averages to the step's exact m'."""
    n = 2048
    _, _, hist = _run(orc, n, 4)
    t, p, g, st = hist[-1]
    m, v = orc.turbo_decode(st, n, t, HY["beta1"], HY["beta2"], HY["eps"])
    _, mexact, vexact, _ = orc.step_fp32(p, g, m, v, t, **HY)
    seeds = 256
    acc = np.zeros(n)
    for s in range(seeds):
        _, st1, _ = orc.turbo_step(p, g, st, t, seed=5000 + s, **HY)
        st1["uscal"] = orc.turbo_finalize(st1["uscal"], n)  # codes decode with their scale
        mnext, _ = orc.turbo_decode(st1, n, t + 1, HY["beta1"], HY["beta2"], HY["eps"])
        acc += mnext
    mbar = acc / seeds
    # elements whose residual lies well inside the code range (+-1.5 encode
    # scales): there the rounding is unbiased, so the mean decoded m regresses
    # on the exact m with slope 1 (a first moment normalised by anything but
    # the persisted v would be off by the ratio of the two denominators)
    bc1, bc2 = 1.0 - HY["beta1"] ** t, 1.0 - HY["beta2"] ** t
    q = mexact / bc1 / (np.sqrt(vexact / bc2) + HY["eps"])
    r = q - np.repeat(q.reshape(-1, 64).mean(axis=1), 64)
    inside = np.abs(r) < 0.75 * float(st["uscal"][1])
    assert inside.sum() > n // 4, inside.sum()
    x, y = mexact[inside].astype(np.float64), mbar[inside]
    slope = float((x * y).sum() / (x * x).sum())
    assert abs(slope - 1.0) < 1.5e-2, slope  # seed-to-seed spread about 0.4 %


def check_means_recentred(orc):
    """Each stored bf16 mean is the mean of q_t over its 64 values rounded to
    bf16, and the decoded q of the next step averages to it over every mean
    block (the recentring preserves it)."""
    n = 64 * 9 + 17
    _, st, hist = _run(orc, n, 5)
    t, p, g, st0 = hist[-1]
    m, v = orc.turbo_decode(st0, n, t, HY["beta1"], HY["beta2"], HY["eps"])
    _, mexact, _, _ = orc.step_fp32(p, g, m, v, t, **HY)
    _, st1, _ = orc.turbo_step(p, g, st0, t, **HY)
    st1["uscal"] = orc.turbo_finalize(st1["uscal"], n)
    bc1 = 1.0 - HY["beta1"] ** t
    bc2 = 1.0 - HY["beta2"] ** t
    mnext, vhat = orc.turbo_decode(st1, n, t + 1, HY["beta1"], HY["beta2"], HY["eps"])
    den = np.sqrt(vhat.astype(np.float64) / np.float32(bc2)) + np.float32(HY["eps"])
    q_exact = mexact.astype(np.float64) / np.float32(bc1) / den
    q_dec = mnext.astype(np.float64) / np.float32(bc1) / den
    mu = (st1["umean"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for k in range(-(-n // 64)):
        sl = slice(64 * k, min(n, 64 * k + 64))
        exact_mean = q_exact[sl].mean()
        # bf16 keeps 8 significant bits: half an ulp is at most 2^-8 relative
        tol = 2 ** -8 * abs(exact_mean) * 1.01 + 1e-6 * np.abs(q_exact[sl]).max()
        assert abs(mu[k] - exact_mean) <= tol, (k, mu[k], exact_mean)
        assert abs(q_dec[sl].mean() - mu[k]) <= 1e-5 * (abs(mu[k]) + st1["uscal"][0]), k


def check_finalize_rotates_scales(orc):
    """The finaliser: decode scale <- encode scale, encode scale <- 1.1 *
    sqrt(accumulator / n), accumulator <- 0; the accumulator is the sum of
    the squared residuals r = q - mu of the step."""
    s = orc.turbo_finalize(np.array([0.25, 0.5, 8.0], np.float32), 32, 1.1)
    assert s[0] == np.float32(0.5) and s[2] == 0.0
    assert s[1] == np.float32(1.1) * np.float32(np.sqrt(np.float32(8.0 / 32)))
    n = 64 * 4
    _, _, hist = _run(orc, n, 3)
    t, p, g, st0 = hist[-1]
    _, st1, _ = orc.turbo_step(p, g, st0, t, **HY)
    m, v = orc.turbo_decode(st0, n, t, HY["beta1"], HY["beta2"], HY["eps"])
    _, mexact, _, _ = orc.step_fp32(p, g, m, v, t, **HY)
    _, vhat = orc.turbo_decode(st1, n, t + 1, HY["beta1"], HY["beta2"], HY["eps"])
    bc1, bc2 = 1.0 - HY["beta1"] ** t, 1.0 - HY["beta2"] ** t
    q = mexact / np.float32(bc1) / (np.sqrt(vhat / np.float32(bc2)) + np.float32(HY["eps"]))
    mu = (st1["umean"].astype(np.uint32) << 16).view(np.float32)
    r = q.astype(np.float64) - np.repeat(mu, 64)[:n]
    assert abs(st1["uscal"][2] - (r ** 2).sum()) <= 1e-5 * (r ** 2).sum(), st1["uscal"][2]


ALL_CHECKS = {
    "uniform_statistics": check_uniform_statistics,
    "counter_is_a_splitmix_position": check_counter_is_a_splitmix_position,
    "two_uniforms_per_output": check_two_uniforms_per_output,
    "q1_grid_closed_forms": check_q1_grid_closed_forms,
    "q1_endpoints": check_q1_endpoints,
    "q1_rounding": check_q1_rounding,
    "ustate_code": check_ustate_code,
    "step_is_adamw_on_decoded_moments": check_step_is_adamw_on_decoded_moments,
    "second_moment_bracketed_and_unbiased": check_second_moment_bracketed_and_unbiased,
    "first_moment_reconstructed": check_first_moment_reconstructed,
    "means_recentred": check_means_recentred,
    "finalize_rotates_scales": check_finalize_rotates_scales,
}
