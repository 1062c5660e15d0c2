"""Pins for the CPU oracle: each check compares the oracle with something other
than itself -- a library routine (numpy binary16, torch bfloat16, torch.bucketize,
numpy.searchsorted, torch.optim.AdamW), textbook rounding in exact arithmetic,
closed forms, brute force on small inputs, or invariants.

Every ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  test_oracle_pins.py runs them on the oracle; test_oracle_mutations.py
runs them on copies of the oracle with a planted mistake and expects a failure.

Sources: "Packed AdamW Reference" README v1.0.0, "The canonical format" (the
E4M11/E4M12 packed word) and the paragraph after it (FP32 update, pack
afterwards); "Packed AdamW / Reference / v1.0.0" code page, "Release scope"
(square the RMS, store afterwards); "TurboAdam" README, "The AdamW update
remains AdamW"; KBench "quantized-optimizer-state" reference.py,
quantized_adamw_step and _requantise.
"""
from __future__ import annotations

import numpy as np

E4M11_MAX = 2.0 - 2.0 ** -11
E4M12_MAX = 2.0 - 2.0 ** -12
HYPER_SETS = [
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01),
    dict(lr=1e-2, beta1=0.8, beta2=0.99, eps=1e-6, wd=0.1),
    dict(lr=3e-4, beta1=0.95, beta2=0.9999, eps=1e-8, wd=0.0),
]


def bits32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32)


def assert_bits_equal(got, exp, what=""):
    g, e = bits32(got), bits32(exp)
    bad = np.nonzero(g != e)[0]
    assert bad.size == 0, (f"{what}: {bad.size} mismatches, first at {bad[:5]}: "
                           f"got {np.asarray(got).reshape(-1)[bad[:5]]} "
                           f"expected {np.asarray(exp).reshape(-1)[bad[:5]]}")


# =========================================================================
# E4 lanes (readings R1-R8 of the oracle header)
# =========================================================================

def check_e4_closed_forms(orc):
    """Largest finite, smallest subnormal, smallest normal, 1.0 and the signed
    zero of each lane, as the IEEE-style layout with bias 15 fixes them."""
    d = orc.e4m11_decode([0x7FFF, 0x0001, 0x0800, 0x07FF, 0x0000, 0x8000, 0xFFFF, 0x7800])
    exp = [E4M11_MAX, 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 0.0, -0.0,
           -E4M11_MAX, 1.0]
    assert_bits_equal(d, exp, "E4M11 closed forms")
    d = orc.e4m12_decode([0xFFFF, 0x0001, 0x1000, 0x0FFF, 0x0000, 0xF000])
    exp = [E4M12_MAX, 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -26, 0.0, 1.0]
    assert_bits_equal(d, exp, "E4M12 closed forms")


def check_e4_shared_binary16_codes(orc):
    """With bias 15 the E4 lanes cover the bottom 16 binades of IEEE binary16
    (subnormals included) with one (E4M11) or two (E4M12) more fraction bits,
    so an E4 code whose extra fraction bits are zero decodes to the binary16
    value with the same sign, exponent and leading fraction bits (numpy's
    binary16 is the library routine)."""
    c = np.arange(65536, dtype=np.uint32)
    ev = c[(c & 1) == 0]
    h = ((ev >> 15) << 15) | (((ev >> 11) & 15) << 10) | ((ev & 0x7FF) >> 1)
    exp = h.astype(np.uint16).view(np.float16).astype(np.float32)
    assert_bits_equal(orc.e4m11_decode(ev.astype(np.uint16)), exp, "E4M11 vs binary16")
    q = c[(c & 3) == 0]
    h = ((q >> 12) << 10) | ((q & 0xFFF) >> 2)
    exp = h.astype(np.uint16).view(np.float16).astype(np.float32)
    assert_bits_equal(orc.e4m12_decode(q.astype(np.uint16)), exp, "E4M12 vs binary16")


def check_e4_equal_spacing_and_sign(orc):
    """Within and across binades the codes between two binary16-shared codes are
    equally spaced (each is the mean of its neighbours), magnitudes increase
    strictly with the code, and the E4M11 sign bit negates the value."""
    m = orc.e4m11_decode(np.arange(32768, dtype=np.uint16)).astype(np.float64)
    assert np.all(np.diff(m) > 0), "E4M11 not strictly increasing"
    odd = np.arange(1, 32767, 2)
    assert np.array_equal(2.0 * m[odd], m[odd - 1] + m[odd + 1]), "E4M11 spacing"
    neg = orc.e4m11_decode((np.arange(32768) | 0x8000).astype(np.uint16))
    assert_bits_equal(neg, -m.astype(np.float32), "E4M11 sign")
    r = orc.e4m12_decode(np.arange(65536, dtype=np.uint16)).astype(np.float64)
    assert np.all(np.diff(r) > 0), "E4M12 not strictly increasing"
    k = np.arange(1, 65535)
    k = k[(k & 3) != 0]
    assert np.array_equal(2.0 * r[k], r[k - 1] + r[k + 1]), "E4M12 spacing"


def check_e4_roundtrip_all_codes(orc):
    """decode -> encode is the identity on all 65,536 codes of each lane
    (including 0x8000 = -0 on the signed lane)."""
    c = np.arange(65536, dtype=np.uint16)
    assert np.array_equal(orc.e4m11_encode(orc.e4m11_decode(c)), c), "E4M11 round trip"
    assert np.array_equal(orc.e4m12_encode(orc.e4m12_decode(c)), c), "E4M12 round trip"


def textbook_round(ax: np.ndarray, mbits: int, maxval: float) -> np.ndarray:
    """Round |x| to nearest on the grid of a float format with ``mbits``
    fraction bits and smallest normal exponent -14, ties to an even multiple of
    the local step (numpy.rint is round-half-even; the scalings are exact in
    float64), then clamp to the largest finite value."""
    ax = np.asarray(ax, np.float64)
    _, ex = np.frexp(ax)
    step = np.ldexp(1.0, np.maximum(ex - 1, -14) - mbits)
    return np.minimum(np.rint(ax / step) * step, maxval)


def _e4_probe_values(orc, rng, count=400_000):
    raw = rng.integers(0, 1 << 32, count, dtype=np.uint64).astype(np.uint32).view(np.float32)
    raw = raw[~np.isnan(raw)]
    logu = (2.0 ** rng.uniform(-30, 1.5, count)) * rng.choice([-1.0, 1.0], count)
    codes = rng.integers(0, 32767, 20000)
    lo = orc.e4m11_decode(codes.astype(np.uint16)).astype(np.float64)
    hi = orc.e4m11_decode((codes + 1).astype(np.uint16)).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)  # exact: <= 14 significant bits
    rcodes = rng.integers(0, 65535, 20000)
    rlo = orc.e4m12_decode(rcodes.astype(np.uint16)).astype(np.float64)
    rhi = orc.e4m12_decode((rcodes + 1).astype(np.uint16)).astype(np.float64)
    rmids = ((rlo + rhi) / 2).astype(np.float32)
    seam = np.array([2.0 ** -14, 2.0 ** -26, 2.0 ** -27, 3 * 2.0 ** -27, 2.0 ** -25,
                     3 * 2.0 ** -26, E4M11_MAX, E4M12_MAX, 2.0, 1e-45, 0.0], np.float32)
    allv = np.concatenate([raw, logu.astype(np.float32), mids, rmids, seam]).astype(np.float32)
    up = np.nextafter(allv, np.float32(np.inf))
    dn = np.nextafter(allv, np.float32(-np.inf))
    out = np.concatenate([allv, up, dn, -allv])
    return out[np.isfinite(out)]


def check_e4_encode_textbook_rne(orc):
    """Encoding rounds to nearest with ties to even and saturates at the largest
    finite value (readings R3, R4), on random values, exact midpoints between
    consecutive codes, their neighbours and the subnormal/normal seam."""
    rng = np.random.default_rng(11)
    x = _e4_probe_values(orc, rng)
    ax = np.abs(x.astype(np.float64))
    exp_m = np.copysign(textbook_round(ax, 11, E4M11_MAX), x).astype(np.float32)
    got_m = orc.e4m11_decode(orc.e4m11_encode(x))
    assert_bits_equal(got_m, exp_m, "E4M11 encode vs textbook RNE")
    exp_r = np.where(x > 0, textbook_round(ax, 12, E4M12_MAX), 0.0).astype(np.float32)
    got_r = orc.e4m12_decode(orc.e4m12_encode(x))
    assert_bits_equal(got_r, exp_r, "E4M12 encode vs textbook RNE")


def check_e4_encode_brute_force(orc):
    """Exhaustive nearest search over all 32,768 E4M11 magnitudes for a few
    thousand values; ties go to the even code; beyond the top, the top."""
    rng = np.random.default_rng(5)
    mags = orc.e4m11_decode(np.arange(32768, dtype=np.uint16)).astype(np.float64)
    x = np.concatenate([
        (2.0 ** rng.uniform(-28, 1.2, 1500)).astype(np.float32),
        ((mags[:-1][::97] + mags[1:][::97]) / 2).astype(np.float32),
    ])
    got = orc.e4m11_encode(x).astype(np.int64) & 0x7FFF
    for xi, gi in zip(x.astype(np.float64), got):
        if xi >= mags[-1]:
            assert gi == 32767
            continue
        dist = np.abs(mags - xi)
        best = np.nonzero(dist == dist.min())[0]
        want = best[0] if best.size == 1 else best[(best % 2) == 0][0]
        assert gi == want, (xi, gi, want)


def check_e4_specials(orc):
    """Saturation (R4), NaN -> +0 (R6), signed zero (R5), unsigned RMS lane (R7)."""
    big = np.array([E4M11_MAX, 2.0, 3.5, 1e30, np.inf, -np.inf, -2.5,
                    np.nextafter(np.float32(E4M11_MAX), np.float32(3))], np.float32)
    assert list(orc.e4m11_encode(big)) == [0x7FFF] * 5 + [0xFFFF, 0xFFFF, 0x7FFF]
    assert list(orc.e4m11_encode([np.nan, -0.0, -1e-30, 1e-30, 0.0])) == [0, 0x8000, 0x8000, 0, 0]
    assert list(orc.e4m12_encode([np.inf, 5.0, np.nan, -1.0, -0.0, -np.inf, 0.0])) == \
        [0xFFFF, 0xFFFF, 0, 0, 0, 0, 0]


# =========================================================================
# binary16 lanes (reading R9) and bfloat16 output
# =========================================================================

def check_fp16_matches_numpy(orc):
    """Inside the finite range the FP16 lanes are IEEE binary16 round to nearest
    even (numpy's conversion), subnormals and -0 included."""
    rng = np.random.default_rng(3)
    allh = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    fin = allh[np.isfinite(allh)]
    s = np.sort(np.unique(fin.astype(np.float64)))
    mids = ((s[:-1] + s[1:]) / 2).astype(np.float32)
    x = np.concatenate([fin, mids, np.nextafter(mids, np.float32(np.inf)),
                        np.nextafter(mids, np.float32(-np.inf)),
                        (rng.uniform(-65519, 65519, 200000)).astype(np.float32),
                        (2.0 ** rng.uniform(-30, 15.9, 200000) *
                         rng.choice([-1, 1], 200000)).astype(np.float32)])
    x = x[np.abs(x) < 65520]
    exp = x.astype(np.float16).view(np.uint16)
    got = orc.fp16_encode(x)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], exp[bad[:5]])
    dec = orc.fp16_decode(np.arange(65536, dtype=np.uint16))
    ok = (bits32(dec) == bits32(allh)) | (np.isnan(dec) & np.isnan(allh))
    assert ok.all(), "binary16 decode"


def check_fp16_specials(orc):
    """Saturation at +-65504 instead of Inf, NaN -> +0 (reading R9)."""
    x = np.array([65504, 65519.99, 65520, 1e9, np.inf, -np.inf, -70000, np.nan], np.float32)
    assert list(orc.fp16_encode(x)) == [0x7BFF] * 5 + [0xFBFF, 0xFBFF, 0]


def check_bf16_matches_torch(orc):
    """The blockwise mode's BF16 output is torch's float32 -> bfloat16
    conversion (round to nearest even, overflow to Inf)."""
    import torch

    rng = np.random.default_rng(9)
    raw = rng.integers(0, 1 << 32, 300000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 1 << 16, 50000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    edge = np.array([0x7F7F8000, 0x7F7F7FFF, 0xFF7F8000, 0x00008000, 0x00018000, 0x7F800000,
                     0x00000001, 0x80000000], np.uint32)
    x = np.concatenate([raw, ties, edge]).view(np.float32)
    got = orc.bf16_round(x)
    exp = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], exp[~nan]), "bfloat16 rounding"
    back = (got[nan].astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(back).all()


# =========================================================================
# The step (all modes): closed forms, torch.optim.AdamW, composition
# =========================================================================

def _step(orc, mode, p, g, st, step, **hy):
    """One step of a mode from its state tuple; returns (p', state', nonfinite)."""
    if mode in ("e4", "fp16"):
        p1, s1, bad = orc.step_packed(p, g, st[0], step, mode=mode, **hy)
        return p1, (s1,), bad
    p1, m1, v1, bad = orc.step_fp32(p, g, st[0], st[1], step, **hy)
    return p1, (m1, v1), bad


def _zero_state(mode, n):
    if mode in ("e4", "fp16"):
        return (np.zeros(n, np.uint32),)
    return (np.zeros(n, np.float32), np.zeros(n, np.float32))


def check_step1_closed_form(orc, mode="e4"):
    """From zero state, step 1 gives m'/bc1 = g and sqrt(v'/bc2) = |g|, so
    p1 = p0 (1 - lr wd) - lr sign(g) / (1 + eps/|g|) up to a few roundings of
    each term; the stored moments are (1-beta1) g and the UNcorrected RMS
    sqrt(1-beta2) |g|, each within half a code step of its lane."""
    rng = np.random.default_rng(21)
    n = 6000
    for hy in HYPER_SETS:
        p0 = rng.normal(0, 1, n).astype(np.float32)
        g = (rng.choice([-1.0, 1.0], n) * 10.0 ** rng.uniform(-7, 0, n)).astype(np.float32)
        p1, st, bad = _step(orc, mode, p0, g, _zero_state(mode, n), 1, **hy)
        assert bad == 0
        a0, ag = p0.astype(np.float64), g.astype(np.float64)
        upd = hy["lr"] * np.sign(ag) / (1.0 + hy["eps"] / np.abs(ag))
        exp = a0 * (1.0 - hy["lr"] * hy["wd"]) - upd
        tol = 2.0 ** -20 * (np.abs(a0) + np.abs(upd))
        err = np.abs(p1.astype(np.float64) - exp)
        assert np.all(err <= tol), f"{mode} step-1 closed form: max err/tol {np.max(err / tol)}"
        m_exact = (1.0 - hy["beta1"]) * ag
        r_exact = np.sqrt(1.0 - hy["beta2"]) * np.abs(ag)
        if mode == "fp32":
            m_dec, v_dec = st
            r_dec = np.sqrt(v_dec.astype(np.float64))
            rel_m, rel_r = 2.0 ** -22, 2.0 ** -22
        else:
            m_dec, r_dec = orc.decode_state(st[0], mode=mode)
            rel_m = 2.0 ** -12 if mode == "e4" else 2.0 ** -11
            rel_r = 2.0 ** -13 if mode == "e4" else 2.0 ** -11
        # below the smallest normal a lane's step is absolute: half of it
        floor_m = {"e4": 2.0 ** -26, "fp16": 2.0 ** -25, "fp32": 0.0}[mode]
        floor_r = {"e4": 2.0 ** -27, "fp16": 2.0 ** -25, "fp32": 0.0}[mode]
        lim_m = E4M11_MAX if mode == "e4" else 65504.0
        sat = np.abs(m_exact) >= lim_m
        em = np.abs(m_dec.astype(np.float64) - m_exact)
        assert np.all((em <= rel_m * np.abs(m_exact) * 1.0001 + floor_m) | sat), \
            f"{mode} stored first moment"
        er = np.abs(np.asarray(r_dec, np.float64) - r_exact)
        assert np.all(er <= rel_r * r_exact * 1.0001 + floor_r), f"{mode} stored RMS"


def check_zero_gradient_pure_decay(orc, mode="e4"):
    """g = 0 (either sign) with zero state: the update term is 0 / eps = 0, so
    p1 = fl(p0 * (1 - lr wd)) exactly and the state stays zero."""
    rng = np.random.default_rng(4)
    n = 3001
    for hy in HYPER_SETS:
        p0 = rng.normal(0, 0.02, n).astype(np.float32)
        g = np.where(rng.random(n) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        p1, st, bad = _step(orc, mode, p0, g, _zero_state(mode, n), 7, **hy)
        assert bad == 0
        assert_bits_equal(p1, p0 * np.float32(1.0 - hy["lr"] * hy["wd"]), f"{mode} decay")
        for s in st:
            assert not np.any(np.asarray(s).view(np.uint32)), f"{mode} state not zero"


def check_fp32_matches_torch_adamw(orc):
    """The FP32 mode follows torch.optim.AdamW (CPU, single-tensor) over many
    steps within rounding; torch orders its operations differently (lerp for
    the first moment, sqrt(v)/sqrt(bc2)), so the comparison has a tolerance."""
    import torch

    rng = np.random.default_rng(8)
    n = 5000
    for hy in HYPER_SETS:
        p = rng.normal(0, 0.02, n).astype(np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        tp = torch.nn.Parameter(torch.from_numpy(p.copy()))
        opt = torch.optim.AdamW([tp], lr=hy["lr"], betas=(hy["beta1"], hy["beta2"]),
                                eps=hy["eps"], weight_decay=hy["wd"], foreach=False,
                                fused=False)
        for t in range(1, 26):
            g = rng.normal(0, 1e-3, n).astype(np.float32)
            p, m, v, _ = orc.step_fp32(p, g, m, v, t, **hy)
            tp.grad = torch.from_numpy(g.copy())
            opt.step()
        st = opt.state[tp]
        np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-6, atol=5e-8)
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=2e-5, atol=3e-10)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=2e-5, atol=1e-16)


def _ieee_sqrt_f32(x):
    """Correctly rounded binary32 square root of a float32 tensor (x >= 0),
    checked: y is the root exactly when x lies between the squares of the
    midpoints from y to its two binary32 neighbours, and both squares are
    exact in binary64 (25-bit factors)."""
    import torch

    y = torch.sqrt(x.double()).float()
    y32 = y.numpy()
    xd, yd = x.double().numpy(), y32.astype(np.float64)
    up = (np.nextafter(y32, np.float32(np.inf)).astype(np.float64) - yd) / 2
    down = (yd - np.nextafter(y32, np.float32(0)).astype(np.float64)) / 2
    pos = yd > 0
    assert np.all((yd[pos] - down[pos]) ** 2 <= xd[pos]), "square root rounded up too far"
    assert np.all(xd[pos] <= (yd[pos] + up[pos]) ** 2), "square root rounded down too far"
    return y


def _page_spec_fp32_step(p, g, m, v, step, lr, beta1, beta2, eps, wd):
    """The FP32 update as KBench "quantized-optimizer-state" reference.py
    (quantized_adamw_step) prints it: torch float32 tensors on the CPU meeting
    Python floats, each operator one float32 rounding, evaluated left to right
    as Python parses it -- so ((1-beta2)*g)*g, ((lr/bc1)*m_new)/denom and
    (p*(1-lr*wd)) - upd.  The scalars (1-beta1, beta2**step, lr/bc1, 1-lr*wd)
    are Python doubles, which torch rounds once to float32 when it meets the
    tensors.

    One exception: torch's CPU square root is not correctly rounded on every
    machine (with AVX-512 it comes out one ulp low for about 0.6 % of binary32
    inputs), while the page's float32 .sqrt() means the IEEE one.  So the root
    is taken in float64 and rounded once to float32 -- the correctly rounded
    binary32 root, since a binary64 result rounded to binary32 is never double
    rounded for the square root of a binary32 operand (S. A. Figueroa, "When is
    double rounding innocuous?", SIGNUM Newsletter 30(3), 1995) -- and each
    root is checked against its exact bracket."""
    import torch

    p, g, m, v = (torch.from_numpy(np.array(a, np.float32)) for a in (p, g, m, v))
    new_m = beta1 * m + (1.0 - beta1) * g
    new_v = beta2 * v + (1.0 - beta2) * g * g
    corr1 = 1.0 - beta1 ** step
    corr2 = 1.0 - beta2 ** step
    den = _ieee_sqrt_f32(new_v / corr2) + eps
    step_size = lr / corr1
    update = step_size * new_m / den
    p_new = p * (1.0 - lr * wd) - update
    return p_new.numpy(), new_m.numpy(), new_v.numpy()


def _adversarial_elements(rng, n):
    """p, g, m, v: typical Adam scales, plus exact zeros of either sign,
    subnormals, huge and tiny magnitudes, and moments that nearly cancel the
    new gradient term (a large share of each kind)."""
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = (rng.choice([-1.0, 1.0], n) * 10.0 ** rng.uniform(-12, 1, n)).astype(np.float32)
    m = (rng.choice([-1.0, 1.0], n) * 10.0 ** rng.uniform(-12, 0, n)).astype(np.float32)
    v = (10.0 ** rng.uniform(-30, 0, n)).astype(np.float32)
    k = n // 10
    g[:k] = np.where(rng.random(k) < 0.5, 0.0, -0.0)
    m[k:2 * k] = np.where(rng.random(k) < 0.5, 0.0, -0.0)
    v[k:2 * k] = 0.0
    sub = np.float32(2.0 ** -126) * rng.random(k).astype(np.float32)
    g[2 * k:3 * k] = sub * rng.choice([-1, 1], k)
    m[3 * k:4 * k] = sub
    v[4 * k:5 * k] = np.abs(sub)
    p[5 * k:6 * k] = sub * 3
    # first-moment cancellation: beta1*m close to -(1-beta1)*g
    m[6 * k:7 * k] = (-g[6 * k:7 * k] / 9.0 * (1 + 1e-6 * rng.normal(size=k))).astype(np.float32)
    # update about as large as the decayed parameter
    p[7 * k:8 * k] = (np.sign(m[7 * k:8 * k]) * 1e-3).astype(np.float32)
    return p, g, m, v


def check_fp32_element_matches_page_spec(orc):
    """The oracle's FP32 element is, bit for bit, the page's own update
    expression evaluated in float32 (torch on the CPU), over typical and
    adversarial inputs (zeros, subnormals, extreme magnitudes, cancellation)
    at early steps and at late steps where 1 - beta2**step rounds to 1."""
    rng = np.random.default_rng(31)
    n = 40000
    for hy in HYPER_SETS:
        for step in (1, 2, 10, 1000, 20000, 10 ** 6):
            p, g, m, v = _adversarial_elements(rng, n)
            ep, em, ev = _page_spec_fp32_step(p, g, m, v, step, **hy)
            op, om, ov, _ = orc.step_fp32(p, g, m, v, step, **hy)
            assert_bits_equal(om, em, f"m' at step {step}")
            assert_bits_equal(ov, ev, f"v' at step {step}")
            assert_bits_equal(op, ep, f"p' at step {step}")


def _random_state_words(rng, n, mode):
    if mode == "e4":
        m = rng.integers(0, 65536, n)
        r = rng.integers(0, 65536, n)
    else:  # finite binary16 codes; RMS lane non-negative
        m = rng.integers(0, 0x7C00, n) | (rng.integers(0, 2, n) << 15)
        r = rng.integers(0, 0x7C00, n)
    return ((r.astype(np.uint64) << 16) | m.astype(np.uint64)).astype(np.uint32)


def check_packed_is_fp32_step_on_decoded_state(orc, mode="e4"):
    """A packed step equals the FP32 step run on the decoded prior state, with
    v = r*r (the square of the stored RMS), followed by packing m' into the low
    lane and sqrt(v') into the high lane."""
    rng = np.random.default_rng(13)
    n = 20000
    for hy in HYPER_SETS:
        w0 = _random_state_words(rng, n, mode)
        if mode == "e4":  # typical Adam-scale moments as well as random codes
            w0[: n // 2], _ = orc.encode_state(rng.normal(0, 1e-3, n // 2),
                                               np.abs(rng.normal(0, 1e-3, n // 2)))
        p0 = rng.normal(0, 0.02, n).astype(np.float32)
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        p1, w1, _ = orc.step_packed(p0, g, w0, 5, mode=mode, **hy)
        m0, r0 = orc.decode_state(w0, mode=mode)
        v0 = r0 * r0
        pf, mf, vf, _ = orc.step_fp32(p0, g, m0, v0, 5, **hy)
        assert_bits_equal(p1, pf, f"{mode} p vs FP32 on decoded state")
        wexp, _ = orc.encode_state(mf, np.sqrt(vf), mode=mode)
        bad = np.nonzero(w1 != wexp)[0]
        assert bad.size == 0, f"{mode} state words: {bad.size} mismatches"


def check_sharding_invariance(orc, mode="e4"):
    """Elements are independent: the step over a concatenation equals the steps
    over its pieces."""
    rng = np.random.default_rng(2)
    n = 9001
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    st = _zero_state(mode, n)
    pa, sa, _ = _step(orc, mode, p, g, st, 3)
    cuts = [0, 1, 4, 1000, 4097, 9001]
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        pb, sb, _ = _step(orc, mode, p[lo:hi], g[lo:hi], tuple(s[lo:hi] for s in st), 3)
        assert_bits_equal(pb, pa[lo:hi])
        for x, y in zip(sb, sa):
            assert np.array_equal(np.asarray(x).view(np.uint32),
                                  np.asarray(y[lo:hi]).view(np.uint32))


def check_nonfinite_count(orc):
    """Non-finite gradients are counted, never repaired: NaN state lanes encode
    to +0, infinite moments saturate (R4, R6)."""
    n = 64
    p = np.full(n, 0.5, np.float32)
    g = np.full(n, 1e-3, np.float32)
    g[[3, 9, 40]] = np.nan
    g[[5, 60]] = np.inf
    p1, w1, bad = orc.step_packed(p, g, np.zeros(n, np.uint32), 1)
    assert bad == 5
    assert list(w1[[3, 9, 40]]) == [0, 0, 0]
    assert list(w1[[5, 60]]) == [0xFFFF7FFF, 0xFFFF7FFF]
    assert np.isnan(p1[[3, 5]]).all() and np.isfinite(p1[[0, 1, 2, 4]]).all()
    p1, w1, bad = orc.step_packed(p, g, np.zeros(n, np.uint32), 1, mode="fp16")
    assert bad == 5 and list(w1[[3, 9, 40]]) == [0, 0, 0]
    assert list(w1[[5, 60]]) == [0x7BFF7BFF, 0x7BFF7BFF]


# =========================================================================
# 8-bit blockwise mode (KBench quantized_adamw_step / _requantise)
# =========================================================================

def _maps():
    import workloads as wl

    return [
        (wl.dynamic_qmap_signed(), True),
        (wl.dynamic_qmap_unsigned(), False),
        (wl.linear_qmap_signed(), True),
        (wl.random_qmap(3, True), True),
        (wl.random_qmap(4, False), False),
    ]


def _requant_inputs(rng, q, signed):
    """Blocks of random values plus blocks holding exact midpoints (absmax 1):
    Adam-scale blocks, a midpoint block, a tiny (~1e-25) block, an all-zero
    block and a short tail."""
    B = 2048
    mid = ((q[:-1] + q[1:]) * np.float32(0.5)).astype(np.float32)
    mids = np.concatenate([mid, np.nextafter(mid, np.float32(2)),
                           np.nextafter(mid, np.float32(-2))])
    b_mid = np.zeros(B, np.float32)
    b_mid[: mids.size] = mids if signed else np.abs(mids)
    b_mid[-1] = 1.0
    x = rng.normal(0, 1e-3, 5 * B).astype(np.float32)
    if not signed:
        x = np.abs(x) ** 2
    tiny = (rng.normal(0, 1e-25, B)).astype(np.float32)
    if not signed:
        tiny = np.abs(tiny)
    return np.concatenate([x, b_mid, tiny, np.zeros(B, np.float32), x[: B // 3]])


def check_requantise_matches_torch_spec(orc):
    """_requantise as the KBench reference states it with torch primitives:
    amax per block, clamp(min=1e-30), bucketize against the 255 midpoints.
    The short last block is zero-padded for torch (|0| never raises a max)."""
    import torch

    rng = np.random.default_rng(17)
    B = 2048
    for q, signed in _maps():
        x = _requant_inputs(rng, q, signed)
        code, amax = orc.requantise(x, q)
        nb = -(-x.size // B)
        xp = np.zeros(nb * B, np.float32)
        xp[: x.size] = x
        tx = torch.from_numpy(xp).view(nb, B)
        tq = torch.from_numpy(q.copy())
        tam = tx.abs().amax(-1)
        c = tx / tam.clamp(min=1e-30).unsqueeze(-1)
        mid = (tq[:-1] + tq[1:]) * 0.5
        tcode = torch.bucketize(c, mid).reshape(-1)[: x.size].numpy()
        assert np.array_equal(code.astype(np.int64), tcode), "codes vs torch spec"
        assert_bits_equal(amax, tam.numpy(), "absmax vs torch spec")


def check_requantise_searchsorted(orc):
    """The code is the number of midpoints strictly below x / max(absmax, 1e-30):
    numpy.searchsorted(side='left') over the binary32 midpoints."""
    rng = np.random.default_rng(19)
    B = 2048
    for q, signed in _maps():
        x = _requant_inputs(rng, q, signed)
        code, amax = orc.requantise(x, q)
        mid = ((q[:-1] + q[1:]) * np.float32(0.5)).astype(np.float32)
        scale = np.maximum(amax, np.float32(1e-30)).astype(np.float32)
        c = (x / np.repeat(scale, B)[: x.size]).astype(np.float32)
        assert np.array_equal(code.astype(np.int64), np.searchsorted(mid, c, side="left"))
        absx = np.abs(x)
        ref = np.array([absx[i:i + B].max() for i in range(0, x.size, B)], np.float32)
        assert_bits_equal(amax, ref, "absmax")


def check_requantise_brute_force_and_invariants(orc):
    """Brute force over the 256 entries: the chosen entry is a nearest one (up
    to the binary32 rounding of midpoints); the element of largest magnitude
    maps to the top (or bottom) entry; an all-zero block stores absmax 0 and the
    entry nearest 0; |decoded| <= absmax."""
    import workloads as wl

    rng = np.random.default_rng(23)
    for q, signed in _maps():
        x = rng.normal(0, 1e-3, 700).astype(np.float32)
        if not signed:
            x = np.abs(x)
        code, amax = orc.requantise(x, q)
        c = x.astype(np.float64) / float(amax[0])
        d = np.abs(c[:, None] - q.astype(np.float64)[None, :])
        best = d.min(axis=1)
        chosen = d[np.arange(x.size), code]
        assert np.all(chosen <= best + 2.0 ** -23), "not a nearest entry"
        k = int(np.argmax(np.abs(x)))
        assert code[k] == (255 if x[k] > 0 else 0)
        assert np.all(np.abs(q[code].astype(np.float64) * amax[0]) <= amax[0])
        zc, za = orc.requantise(np.zeros(2048 + 5, np.float32), q)
        assert np.all(za == 0) and np.all(zc == wl.nearest_zero_code(q))


def check_blockwise_step_composition(orc):
    """quantized_adamw_step: dequantise (map entry x block absmax, binary32
    multiply), the FP32 AdamW element update, BF16 parameter output (torch
    conversion) and requantisation of the new moments; tails of odd length."""
    import torch
    import workloads as wl

    rng = np.random.default_rng(29)
    q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
    for n in (2048 * 3 + 777, 1, 2048):
        nb = -(-n // 2048)
        p = rng.normal(0, 0.02, n).astype(np.float32)
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        mc = rng.integers(0, 256, n).astype(np.uint8)
        vc = rng.integers(0, 256, n).astype(np.uint8)
        ma = np.abs(rng.normal(0, 1e-3, nb)).astype(np.float32)
        va = np.abs(rng.normal(0, 1e-6, nb)).astype(np.float32)
        for hy in HYPER_SETS[:2]:
            pb, mc1, ma1, vc1, va1, _ = orc.step_blockwise8(p, g, mc, ma, vc, va, q1, q2, 4,
                                                            **hy)
            m = q1[mc] * np.repeat(ma, 2048)[:n]
            v = q2[vc] * np.repeat(va, 2048)[:n]
            pf, mf, vf, _ = orc.step_fp32(p, g, m, v, 4, **hy)
            exp_pb = torch.from_numpy(pf).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(pb, exp_pb.view(np.uint16)), "bf16 p"
            ec, ea = orc.requantise(mf, q1)
            assert np.array_equal(mc1, ec) and np.array_equal(bits32(ma1), bits32(ea))
            ec, ea = orc.requantise(vf, q2)
            assert np.array_equal(vc1, ec) and np.array_equal(bits32(va1), bits32(ea))


def check_blockwise_tail_is_zero_padding(orc):
    """A short last block behaves like the same block zero-padded to 2048."""
    import workloads as wl

    rng = np.random.default_rng(31)
    q = wl.dynamic_qmap_signed()
    x = rng.normal(0, 1e-3, 2048 + 513).astype(np.float32)
    xp = np.concatenate([x, np.zeros(2048 - 513, np.float32)])
    c1, a1 = orc.requantise(x, q)
    c2, a2 = orc.requantise(xp, q)
    assert np.array_equal(c1, c2[: x.size]) and np.array_equal(bits32(a1), bits32(a2))


ALL_CHECKS = {
    "e4_closed_forms": check_e4_closed_forms,
    "e4_shared_binary16_codes": check_e4_shared_binary16_codes,
    "e4_equal_spacing_and_sign": check_e4_equal_spacing_and_sign,
    "e4_roundtrip_all_codes": check_e4_roundtrip_all_codes,
    "e4_encode_textbook_rne": check_e4_encode_textbook_rne,
    "e4_encode_brute_force": check_e4_encode_brute_force,
    "e4_specials": check_e4_specials,
    "fp16_matches_numpy": check_fp16_matches_numpy,
    "fp16_specials": check_fp16_specials,
    "bf16_matches_torch": check_bf16_matches_torch,
    "step1_closed_form_e4": lambda o: check_step1_closed_form(o, "e4"),
    "step1_closed_form_fp16": lambda o: check_step1_closed_form(o, "fp16"),
    "step1_closed_form_fp32": lambda o: check_step1_closed_form(o, "fp32"),
    "zero_gradient_decay_e4": lambda o: check_zero_gradient_pure_decay(o, "e4"),
    "zero_gradient_decay_fp16": lambda o: check_zero_gradient_pure_decay(o, "fp16"),
    "zero_gradient_decay_fp32": lambda o: check_zero_gradient_pure_decay(o, "fp32"),
    "fp32_matches_torch_adamw": check_fp32_matches_torch_adamw,
    "fp32_element_matches_page_spec": check_fp32_element_matches_page_spec,
    "packed_e4_is_fp32_on_decoded": lambda o: check_packed_is_fp32_step_on_decoded_state(o, "e4"),
    "packed_fp16_is_fp32_on_decoded":
        lambda o: check_packed_is_fp32_step_on_decoded_state(o, "fp16"),
    "sharding_invariance_e4": lambda o: check_sharding_invariance(o, "e4"),
    "sharding_invariance_fp32": lambda o: check_sharding_invariance(o, "fp32"),
    "nonfinite_count": check_nonfinite_count,
    "requantise_matches_torch_spec": check_requantise_matches_torch_spec,
    "requantise_searchsorted": check_requantise_searchsorted,
    "requantise_brute_force_and_invariants": check_requantise_brute_force_and_invariants,
    "blockwise_step_composition": check_blockwise_step_composition,
    "blockwise_tail_is_zero_padding": check_blockwise_tail_is_zero_padding,
}
