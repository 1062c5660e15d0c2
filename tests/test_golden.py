"""The oracle against stored fixtures (CPU only).

e4_format_constants.json holds the E4 lane constants that follow from the
readings of "Packed AdamW Reference" README, "The canonical format" (IEEE-style
layout, bias 15, no Inf/NaN codes).  single4096_trajectory.json was written by
tests/golden/make_golden.py from the oracle; it guards against an unnoticed
change of the oracle's arithmetic.
"""
import hashlib
import json
import os

import numpy as np

import oracle
import workloads as wl

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_format_constants():
    with open(os.path.join(HERE, "e4_format_constants.json")) as f:
        c = json.load(f)
    for lane, dec, enc in (("e4m11", oracle.e4m11_decode, oracle.e4m11_encode),
                           ("e4m12", oracle.e4m12_decode, oracle.e4m12_encode)):
        top = 0x7FFF if lane == "e4m11" else 0xFFFF
        assert dec([top])[0] == c[lane]["max_finite"]
        assert dec([1])[0] == c[lane]["min_subnormal"]
        assert enc([1.0])[0] == c[lane]["code_of_one"]
        assert enc([c[lane]["min_normal"]])[0] == (0x800 if lane == "e4m11" else 0x1000)
    assert oracle.e4m11_encode([-0.0])[0] == c["e4m11"]["code_of_minus_zero"]
    assert oracle.fp16_encode([1e6])[0] == c["fp16_saturation"]["code"]


def test_single4096_trajectory():
    with open(os.path.join(HERE, "single4096_trajectory.json")) as f:
        doc = json.load(f)
    n, hy = 4096, wl.HYPER
    p0 = wl.normal_np(n, 0.02, 0)
    for mode, steps in doc["modes"].items():
        p = p0.copy()
        st = [np.zeros(n, np.uint32)] if mode != "fp32" else [np.zeros(n, np.float32)] * 2
        for rec in steps:
            t = rec["step"]
            g = wl.normal_np(n, 1e-3, 1000 + t)
            if mode == "fp32":
                p, m, v, bad = oracle.step_fp32(p, g, st[0], st[1], t, **hy)
                st = [m, v]
            else:
                p, s, bad = oracle.step_packed(p, g, st[0], t, mode=mode, **hy)
                st = [s]
            h = hashlib.sha256()
            for a in (p, *st):
                h.update(np.ascontiguousarray(a).tobytes())
            assert bad == rec["nonfinite"]
            assert [int(x) for x in p[:8].view(np.uint32)] == rec["p_head_bits"], (mode, t)
            assert h.hexdigest() == rec["sha256"], (mode, t)
