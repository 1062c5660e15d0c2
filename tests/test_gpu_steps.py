"""GPU AdamW steps against the CPU oracle, bit for bit, through the C ABI.

The packed E4 step ("Packed AdamW / Reference / v1.0.0", "Release scope"),
the FP16-first/FP16-RMS and FP32 comparison modes ("Packed AdamW Reference"
README v1.0.0), one launch per tensor and one launch per tensor list
("Execution contract").  Sizes span several 4096-element chunks with ragged
tails; views start at every 4-byte offset (the 16-byte path peels a head) or
at mismatched offsets (the 4-byte path).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_same_bits, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu

HY = wl.HYPER
# 1_500_007: a launch of a few full tiles per SM with a ragged tail
SIZES = [1, 3, 4, 5, 255, 4095, 4096, 4097, 3 * 4096 + 7, 6143, 6144, 6147, 2 * 6144 + 5, 100_003,
         1_500_007]


@pytest.fixture(scope="module")
def pa():
    import adamw_update_gb300

    return adamw_update_gb300


def _run_packed(pa, mode, p, gs, state, offsets=(0, 0, 0), hy=HY, first_step=1):
    """Run len(gs) steps on the GPU (views at the given element offsets)."""
    import torch

    n = p.size
    bufs = [torch.zeros(n + 8, dtype=dt, device="cuda")
            for dt in (torch.float32, torch.float32, torch.int32)]
    dp, dg, ds = (b[o:o + n] for b, o in zip(bufs, offsets))
    dp.copy_(dev(p))
    ds.copy_(dev(state))
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = pa.pa_adamw_step_packed_e4 if mode == "e4" else pa.pa_adamw_step_packed_fp16
    for k, g in enumerate(gs):
        dg.copy_(dev(g))
        fn(dp, dg, ds, first_step + k, nonfinite=bad, **hy)
    torch.cuda.synchronize()
    return host_f32(dp), host_u32(ds), int(bad.item())


def _oracle_packed(mode, p, gs, state, hy=HY, first_step=1):
    bad = 0
    for k, g in enumerate(gs):
        p, state, b = oracle.step_packed(p, g, state, first_step + k, mode=mode, **hy)
        bad += b
    return p, state, bad


@pytest.mark.parametrize("mode", ["e4", "fp16"])
@pytest.mark.parametrize("n", SIZES)
def test_packed_step_sizes(pa, mode, n):
    rng = np.random.default_rng(n)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    gs = [rng.normal(0, 1e-3, n).astype(np.float32) for _ in range(3)]
    st = np.zeros(n, np.uint32)
    gp, gw, gb = _run_packed(pa, mode, p, gs, st)
    ep, ew, eb = _oracle_packed(mode, p, gs, st)
    assert_same_bits(gp, ep, f"{mode} p n={n}")
    assert_same_bits(gw, ew, f"{mode} state n={n}")
    assert gb == eb == 0


@pytest.mark.parametrize("offsets", [(1, 1, 1), (2, 2, 2), (3, 3, 3), (1, 2, 3), (0, 1, 0)])
def test_packed_e4_misaligned_views(pa, offsets):
    n = 2 * 4096 + 13
    rng = np.random.default_rng(sum(offsets))
    p = rng.normal(0, 0.02, n).astype(np.float32)
    gs = [rng.normal(0, 1e-3, n).astype(np.float32) for _ in range(2)]
    st, _ = oracle.encode_state(rng.normal(0, 1e-3, n), np.abs(rng.normal(0, 1e-3, n)))
    gp, gw, _ = _run_packed(pa, "e4", p, gs, st, offsets)
    ep, ew, _ = _oracle_packed("e4", p, gs, st)
    assert_same_bits(gp, ep, f"p offsets={offsets}")
    assert_same_bits(gw, ew, f"state offsets={offsets}")


def test_single_4096_ten_steps(pa):
    """The single-tensor workload: 4,096 parameters, fresh g each step, 10 steps."""
    n = 4096
    p = wl.normal_np(n, 0.02, 0)
    gs = [wl.normal_np(n, 1e-3, 1000 + t) for t in range(1, 11)]
    st = np.zeros(n, np.uint32)
    for mode in ("e4", "fp16"):
        gp, gw, _ = _run_packed(pa, mode, p, gs, st)
        ep, ew, _ = _oracle_packed(mode, p, gs, st)
        assert_same_bits(gp, ep, f"{mode} p")
        assert_same_bits(gw, ew, f"{mode} state")


@pytest.mark.parametrize("hy", [dict(lr=1e-2, beta1=0.8, beta2=0.99, eps=1e-6, wd=0.1),
                                dict(lr=3e-4, beta1=0.0, beta2=0.0, eps=0.0, wd=0.0),
                                dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)])
def test_packed_e4_random_state_hyper_and_late_steps(pa, hy):
    """Random prior state words (every code reachable), other hyperparameters,
    late global steps (bias corrections near 1)."""
    n = 50_001
    rng = np.random.default_rng(5)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    gs = [rng.normal(0, 1e-3, n).astype(np.float32) for _ in range(2)]
    gp, gw, gb = _run_packed(pa, "e4", p, gs, st, hy=hy, first_step=999)
    ep, ew, eb = _oracle_packed("e4", p, gs, st, hy=hy, first_step=999)
    assert_same_bits(gp, ep, "p")
    assert_same_bits(gw, ew, "state")
    assert gb == eb


def test_nonfinite_gradients_counted(pa):
    n = 5000
    rng = np.random.default_rng(9)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    g[[0, 17, 4096]] = np.nan
    g[[5, 4999]] = np.inf
    g[[6]] = -np.inf
    g[[7]] = 3e38  # finite, but v' overflows
    st = np.zeros(n, np.uint32)
    for mode in ("e4", "fp16"):
        gp, gw, gb = _run_packed(pa, mode, p, [g], st)
        ep, ew, eb = _oracle_packed(mode, p, [g], st)
        assert gb == eb == 7
        nan = np.isnan(ep)
        assert np.array_equal(np.isnan(gp), nan)
        assert_same_bits(gp[~nan], ep[~nan], f"{mode} p")
        assert_same_bits(gw, ew, f"{mode} state")


@pytest.mark.parametrize("n", [1, 4097, 100_003])
def test_fp32_step(pa, n):
    import torch

    rng = np.random.default_rng(n + 1)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    m = rng.normal(0, 1e-4, n).astype(np.float32)
    v = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
    dp, dm, dv = dev(p), dev(m), dev(v)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in range(1, 4):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        pa.pa_adamw_step_fp32(dp, dev(g), dm, dv, t, nonfinite=bad, **HY)
        p, m, v, _ = oracle.step_fp32(p, g, m, v, t, **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(dp), p, "p")
    assert_same_bits(host_f32(dm), m, "m")
    assert_same_bits(host_f32(dv), v, "v")
    assert int(bad.item()) == 0


def _tensors(sizes, rng, mode):
    out = []
    for n in sizes:
        p = rng.normal(0, 0.02, n).astype(np.float32)
        if mode == "fp32":
            out.append([p, np.zeros(n, np.float32), np.zeros(n, np.float32)])
        else:
            out.append([p, np.zeros(n, np.uint32)])
    return out


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_multi_tensor_list_ragged(pa, mode):
    """Empty, tiny and chunk-straddling tensors, views at odd offsets, in one
    launch; equals the oracle tensor by tensor."""
    import torch

    sizes = [0, 1, 3, 4096, 5, 0, 9000, 4097, 2, 30_000]
    rng = np.random.default_rng(3)
    host = _tensors(sizes, rng, mode)
    devs = []
    for k, h in enumerate(host):
        off = k % 4
        views = []
        for a in h:
            dt = torch.int32 if a.dtype == np.uint32 else torch.float32
            buf = torch.zeros(a.size + 8, dtype=dt, device="cuda")
            v = buf[off:off + a.size]
            v.copy_(dev(a)) if a.size else None
            views.append(v)
        devs.append(views)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = {"e4": pa.pa_adamw_step_packed_e4_multi, "fp16": pa.pa_adamw_step_packed_fp16_multi,
          "fp32": pa.pa_adamw_step_fp32_multi}[mode]
    for t in range(1, 4):
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n in sizes]
        dgs = [dev(g) for g in gs]
        entries = [(d[0], dg, *d[1:]) for d, dg in zip(devs, dgs)]
        fn(entries, t, nonfinite=bad, **HY)
        for h, g in zip(host, gs):
            if mode == "fp32":
                h[0], h[1], h[2], _ = oracle.step_fp32(h[0], g, h[1], h[2], t, **HY)
            else:
                h[0], h[1], _ = oracle.step_packed(h[0], g, h[1], t, mode=mode, **HY)
        torch.cuda.synchronize()
    for k, (h, d) in enumerate(zip(host, devs)):
        assert_same_bits(host_f32(d[0]), h[0], f"tensor {k} p")
        for a, dd in zip(h[1:], d[1:]):
            got = host_u32(dd) if a.dtype == np.uint32 else host_f32(dd)
            assert_same_bits(got, a, f"tensor {k} state")
    assert int(bad.item()) == 0


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
@pytest.mark.parametrize("n,off", [(1, 0), (6143, 1), (6145, 3), (3 * 6144 + 7, 2)])
def test_one_tensor_list_with_a_new_gradient_buffer_every_step(pa, mode, n, off):
    """A one-tensor list is passed by value (no descriptor table); each step
    brings a gradient buffer at a new address, as a training loop that
    reallocates its gradients does.  Equals the oracle bit for bit."""
    import torch

    rng = np.random.default_rng(n + off)
    host = _tensors([n], rng, mode)[0]
    views = []
    for a in host:
        dt = torch.int32 if a.dtype == np.uint32 else torch.float32
        buf = torch.zeros(n + 8, dtype=dt, device="cuda")
        views.append(buf[off:off + n])
        views[-1].copy_(dev(a))
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = {"e4": pa.pa_adamw_step_packed_e4_multi, "fp16": pa.pa_adamw_step_packed_fp16_multi,
          "fp32": pa.pa_adamw_step_fp32_multi}[mode]
    keep = []
    for t in range(1, 5):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        gbuf = torch.zeros(n + 8 + t, dtype=torch.float32, device="cuda")
        dg = gbuf[off:off + n]
        dg.copy_(dev(g))
        keep.append(gbuf)  # every step's buffer at its own address
        fn([(views[0], dg, *views[1:])], t, nonfinite=bad, **HY)
        if mode == "fp32":
            host[0], host[1], host[2], _ = oracle.step_fp32(host[0], g, host[1], host[2], t, **HY)
        else:
            host[0], host[1], _ = oracle.step_packed(host[0], g, host[1], t, mode=mode, **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(views[0]), host[0], "p")
    for a, d in zip(host[1:], views[1:]):
        got = host_u32(d) if a.dtype == np.uint32 else host_f32(d)
        assert_same_bits(got, a, "state")
    assert int(bad.item()) == 0


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_multi_tensor_list_longer_than_the_shared_table(pa, mode):
    """600 tensors (more than the 512 descriptors the staged kernel copies into
    shared memory, so the producer walks the table in global memory): sizes
    from 0 to two tiles, views at every 4-byte phase; equals the oracle."""
    import torch

    rng = np.random.default_rng(11)
    sizes = [int(x) for x in rng.choice([0, 1, 3, 4, 7, 100, 6143, 6144, 6149, 12_300], 600)]
    host = _tensors(sizes, rng, mode)
    devs = []
    for k, h in enumerate(host):
        off = (k // 3) % 4
        views = []
        for a in h:
            dt = torch.int32 if a.dtype == np.uint32 else torch.float32
            buf = torch.zeros(a.size + 8, dtype=dt, device="cuda")
            v = buf[off:off + a.size]
            v.copy_(dev(a)) if a.size else None
            views.append(v)
        devs.append(views)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = {"e4": pa.pa_adamw_step_packed_e4_multi, "fp16": pa.pa_adamw_step_packed_fp16_multi,
          "fp32": pa.pa_adamw_step_fp32_multi}[mode]
    for t in (1, 2):
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n in sizes]
        dgs = [dev(g) for g in gs]
        fn([(d[0], dg, *d[1:]) for d, dg in zip(devs, dgs)], t, nonfinite=bad, **HY)
        for h, g in zip(host, gs):
            if mode == "fp32":
                h[0], h[1], h[2], _ = oracle.step_fp32(h[0], g, h[1], h[2], t, **HY)
            else:
                h[0], h[1], _ = oracle.step_packed(h[0], g, h[1], t, mode=mode, **HY)
    torch.cuda.synchronize()
    for k, (h, d) in enumerate(zip(host, devs)):
        assert_same_bits(host_f32(d[0]), h[0], f"tensor {k} p")
        for a, dd in zip(h[1:], d[1:]):
            got = host_u32(dd) if a.dtype == np.uint32 else host_f32(dd)
            assert_same_bits(got, a, f"tensor {k} state")
    assert int(bad.item()) == 0


def test_multi_gpt52_equals_oracle(pa):
    """The 52-tensor GPT list (9,677,312 parameters), packed E4, 2 steps."""
    import torch

    sizes = [n for _, n in wl.GPT52_SHAPES]
    total = sum(sizes)
    flat_p = torch.empty(total, dtype=torch.float32, device="cuda")
    wl.fill_normal_(flat_p, 0.02, seed=0)
    flat_g = torch.empty(total, dtype=torch.float32, device="cuda")
    flat_s = torch.zeros(total, dtype=torch.int32, device="cuda")
    p_host = host_f32(flat_p).copy()
    s_host = np.zeros(total, np.uint32)
    offs = np.cumsum([0] + sizes)
    for t in range(1, 3):
        wl.fill_normal_(flat_g, 1e-3, seed=t, stream=5)
        entries = [(flat_p[a:b], flat_g[a:b], flat_s[a:b]) for a, b in zip(offs[:-1], offs[1:])]
        pa.pa_adamw_step_packed_e4_multi(entries, t, **HY)
        p_host, s_host, _ = oracle.step_packed(p_host, host_f32(flat_g), s_host, t, threads=8, **HY)
    torch.cuda.synchronize()
    assert_same_bits(host_f32(flat_p), p_host, "gpt-52 p")
    assert_same_bits(host_u32(flat_s), s_host, "gpt-52 state")


def test_multi_equals_single_and_is_shard_invariant(pa):
    """A list over pieces of one tensor (cut at arbitrary points) gives the same
    bits as the single-tensor call over the whole (elementwise independence)."""
    import torch

    n = 70_001
    rng = np.random.default_rng(12)
    p = dev(rng.normal(0, 0.02, n).astype(np.float32))
    g = dev(rng.normal(0, 1e-3, n).astype(np.float32))
    s = dev(rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32))
    p2, s2 = p.clone(), s.clone()
    pa.pa_adamw_step_packed_e4(p, g, s, 3, **HY)
    cuts = [0, 1, 6, 4096, 4101, 33_333, n]
    pa.pa_adamw_step_packed_e4_multi(
        [(p2[a:b], g[a:b], s2[a:b]) for a, b in zip(cuts[:-1], cuts[1:])], 3, **HY)
    torch.cuda.synchronize()
    assert torch.equal(p, p2) and torch.equal(s, s2)


def test_argument_errors(pa):
    import torch

    x = torch.zeros(8, dtype=torch.float32, device="cuda")
    w = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PackedAdamError):
        pa.pa_adamw_step_packed_e4(x, x, w, 0)
    with pytest.raises(pa.PackedAdamError):
        pa.pa_adamw_step_packed_e4(x, x, w, 1, beta1=1.0)
    with pytest.raises(pa.PackedAdamError):
        pa.pa_adamw_step_packed_e4(x, x, w, 1, lr=float("nan"))
    with pytest.raises(pa.PackedAdamError):
        pa.pa_adamw_step_packed_e4(x[1:].view(-1), x[1:], w[1:], 1,
                                   nonfinite=int(x.data_ptr()) + 4)
    raw = x.data_ptr() + 2  # not 4-byte aligned
    assert pa._lib.pa_adamw_step_packed_e4(raw, raw, raw, 4, 1, 1e-3, .9, .999, 1e-8, 0,
                                           None, None) == 3


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_late_steps_unit_bias_correction(pa, mode):
    """Global steps where 1 - beta2^step rounds to 1.0f take the kernel
    instantiation that skips v'/bc2; the bits must not change."""
    import torch

    n = 9001
    rng = np.random.default_rng(21)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    gs = [rng.normal(0, 1e-3, n).astype(np.float32) for _ in range(2)]
    assert oracle.hyperparams(100_000, **HY)[4] == 1.0  # bc2
    if mode == "fp32":
        m = rng.normal(0, 1e-4, n).astype(np.float32)
        v = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
        dp, dm, dv = dev(p), dev(m), dev(v)
        for k, g in enumerate(gs):
            pa.pa_adamw_step_fp32_multi([(dp, dev(g), dm, dv)], 100_000 + k, **HY)
            p, m, v, _ = oracle.step_fp32(p, g, m, v, 100_000 + k, **HY)
        torch.cuda.synchronize()
        assert_same_bits(host_f32(dp), p, "p")
        assert_same_bits(host_f32(dm), m, "m")
        assert_same_bits(host_f32(dv), v, "v")
        return
    st = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    if mode == "fp16":
        st = (st & 0x7BFF7BFF).astype(np.uint32)
    gp, gw, gb = _run_packed(pa, mode, p, gs, st, first_step=100_000)
    ep, ew, eb = _oracle_packed(mode, p, gs, st, first_step=100_000)
    assert_same_bits(gp, ep, f"{mode} p")
    assert_same_bits(gw, ew, f"{mode} state")
    assert gb == eb


def test_no_pipeline_fault_after_the_steps(pa):
    """The staged kernels' bounded waits never ran out during this module."""
    assert pa.pa_device_fault(clear=True) == 0


@pytest.mark.parametrize("first_step", [1, 100_000])
@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_large_launch_sampled(pa, mode, first_step):
    """A launch of at least 32 tiles per CTA (4,864 tiles of 6,144 elements on
    a 152-SM GB300) takes the kernel instantiation whose whole tiles keep the
    branch-free arithmetic one lane at a time; smaller launches pair it.  One
    tensor of 30,000,013 elements with random prior state, two steps at early
    and at late global steps (1 - beta2^step rounding to 1.0f takes the
    instantiation that skips v'/bc2), 0.1 % zero gradients (warps whose share
    holds one take the per-vector path); 16 slices of 4,096 elements (the
    ragged end included) advanced by the oracle must match bit for bit
    (elements are independent)."""
    import torch

    n = 30_000_013
    rng = np.random.default_rng(first_step + len(mode))
    starts = sorted(set(rng.integers(0, n - 4096, 15).tolist()) | {n - 4096})
    p = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).cuda()
    if mode == "fp32":
        state = [torch.from_numpy(rng.normal(0, 1e-4, n).astype(np.float32)).cuda(),
                 torch.from_numpy((rng.normal(0, 1e-3, n) ** 2).astype(np.float32)).cuda()]
    else:
        w = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        if mode == "fp16":
            w &= np.uint32(0x7BFF7BFF)
        state = [torch.from_numpy(w.view(np.int32)).cuda()]
    host = [[p[a:a + 4096].cpu().numpy()] + [s[a:a + 4096].cpu().numpy() for s in state]
            for a in starts]
    if mode != "fp32":
        for h in host:
            h[1] = h[1].view(np.uint32)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in (first_step, first_step + 1):
        gn = rng.normal(0, 1e-3, n).astype(np.float32)
        gn[rng.random(n) < 1e-3] = 0.0  # about a quarter of the warps' shares take the per-vector path
        g = torch.from_numpy(gn).cuda()
        if mode == "fp32":
            pa.pa_adamw_step_fp32(p, g, state[0], state[1], t, nonfinite=bad, **HY)
        else:
            fn = pa.pa_adamw_step_packed_e4 if mode == "e4" else pa.pa_adamw_step_packed_fp16
            fn(p, g, state[0], t, nonfinite=bad, **HY)
        gh = [g[a:a + 4096].cpu().numpy() for a in starts]
        for h, gs in zip(host, gh):
            if mode == "fp32":
                h[0], h[1], h[2], _ = oracle.step_fp32(h[0], gs, h[1], h[2], t, **HY)
            else:
                h[0], h[1], _ = oracle.step_packed(h[0], gs, h[1], t, mode=mode, **HY)
    torch.cuda.synchronize()
    for a, h in zip(starts, host):
        assert_same_bits(p[a:a + 4096].cpu().numpy(), h[0], f"{mode} p at {a}")
        for s, e in zip(state, h[1:]):
            got = s[a:a + 4096].cpu().numpy()
            got = got.view(np.uint32) if mode != "fp32" else got
            assert_same_bits(got, e, f"{mode} state at {a}")
