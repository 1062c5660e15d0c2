"""The seeded input generators (workloads/), on the CPU: reproducible, and
with the distributions of the workloads they stand in for (g ~ N(0, 1e-3);
1e-3 * t(df=3) with 1e-4 of the entries boosted 1e4-fold for the flat
workload; per-tensor scales 10^U(-5,-1) and 1 % exact zeros for the GPT-2
list)."""
import numpy as np
import pytest

import workloads as wl

torch = pytest.importorskip("torch")


def test_normal_is_reproducible_and_scaled():
    a = wl.fill_normal_(torch.empty(1 << 20), 1e-3, seed=5)
    b = wl.fill_normal_(torch.empty(1 << 20), 1e-3, seed=5)
    c = wl.fill_normal_(torch.empty(1 << 20), 1e-3, seed=5, stream=1)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert abs(float(a.std()) / 1e-3 - 1.0) < 0.01
    assert abs(float(a.mean())) < 5e-6


def test_student_t_with_saturating_boost():
    n = 1 << 23
    g = wl.fill_student_t_saturating_(torch.empty(n), seed=3).double()
    a = g.abs()
    # t(3) has median |t| = 0.7649; the boosted 1e-4 barely moves the median
    assert abs(float(a.median()) / 1e-3 / 0.7649 - 1.0) < 0.02
    # boosted entries are 10 * t3 in size: |g| > 0.05 unless |t3| < 0.005,
    # while unboosted ones reach 0.05 only for |t3| > 50 (probability ~2e-5)
    big = int((a > 0.05).sum())
    assert 0.8e-4 * n < big < 1.3e-4 * n, big
    # heavy tails: P(|t3| > 5) = 0.0154
    tail = float((a > 5e-3).double().mean())
    assert abs(tail / 0.0154 - 1.0) < 0.1, tail
    again = wl.fill_student_t_saturating_(torch.empty(n), seed=3)
    assert torch.equal(again, g.float())


def test_gpt2_gradients_scales_and_zeros():
    sizes = [1 << 18, 1 << 17, 3 * (1 << 16), 768]
    g = wl.fill_gpt2_grads_(torch.empty(sum(sizes)), sizes, seed=11)
    off = 0
    for n in sizes:
        seg = g[off:off + n].double()
        off += n
        zero = float((seg == 0).double().mean())
        nz = seg[seg != 0]
        s = float(nz.std())
        assert 1e-5 * 0.9 <= s <= 1e-1 * 1.1
        if n >= 1 << 16:
            assert abs(zero / 0.01 - 1.0) < 0.15, zero
    again = wl.fill_gpt2_grads_(torch.empty(sum(sizes)), sizes, seed=11)
    assert torch.equal(again, g)


def test_blockwise_initial_codes_and_blocks():
    q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
    assert q1[wl.nearest_zero_code(q1)] == 0.0 and q2[wl.nearest_zero_code(q2)] == 0.0
    assert wl.blocks(1) == 1 and wl.blocks(2048) == 1 and wl.blocks(2049) == 2
    assert wl.blocks(10 ** 9) == 488_282
    assert np.all(np.diff(q1) > 0) and q1[0] == -1.0 and q1[-1] == 1.0
    assert np.all(np.diff(q2) > 0) and q2[0] == 0.0 and q2[-1] == 1.0
