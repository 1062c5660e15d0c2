"""Parity at the full workload sizes, in the launch configuration bench.py
times (one multi-tensor launch per step over the workload's tensor list).

flat-7e9: 7e9 parameters (84 GB on the device); 64 chunks of 2^20 elements
are copied out before and after each of two steps -- seeded positions, the
last (ragged) chunk, and chunks holding saturating gradients -- and the oracle
advances exactly those elements, which must match bit for bit (elements are
independent).  A full-array device check counts non-finite values and the
state codes at the finite bound.
gpt2-148: all 124,439,808 parameters, packed E4 and FP16, two steps, in full.
blockwise-1e9: 64 sampled 2048-blocks (the short last block included).
turbo-124m: 48 sampled slices of eight 128-value blocks over three steps.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_same_bits, assert_same_f32_nan_aware

pytestmark = pytest.mark.gpu

CH = 1 << 20


@pytest.fixture(scope="module")
def pa():
    import adamw_update_gb300

    return adamw_update_gb300


def _bench():
    import bench

    return bench


def test_flat_7e9_sampled(pa):
    import torch

    b = _bench()
    w = b.Workload("flat-7e9", "e4", torch.device("cuda"), seed=1234)
    n = w.n
    nonfinite = torch.zeros(1, dtype=torch.int64, device="cuda")
    run = b.step_fn(pa, w, wl.HYPER, nonfinite)
    rng = np.random.default_rng(77)
    nchunks = -(-n // CH)
    big = torch.nonzero(w.g[: 64 * CH].abs() > 0.5).flatten()[:8].cpu().numpy() // CH
    picks = sorted(set(rng.integers(0, nchunks - 1, 52).tolist()) | set(big.tolist())
                   | {0, nchunks - 1})[:64]
    ranges = [(c * CH, min(n, (c + 1) * CH)) for c in picks]
    host = [[w.p[a:e].cpu().numpy(), w.g[a:e].cpu().numpy(),
             w.s[0][a:e].cpu().numpy().view(np.uint32)] for a, e in ranges]
    for t in (1, 2):
        run(t)
        torch.cuda.synchronize()
        for (a, e), h in zip(ranges, host):
            h[0], h[2], _ = oracle.step_packed(h[0], h[1], h[2], t, threads=8, **wl.HYPER)
            assert_same_bits(w.p[a:e].cpu().numpy(), h[0], f"p [{a}, {e}) step {t}")
            assert_same_bits(w.s[0][a:e].cpu().numpy().view(np.uint32), h[2],
                             f"state [{a}, {e}) step {t}")
    assert int(nonfinite.item()) == 0
    assert not torch.isnan(w.p).any().item()
    sat = ((w.s[0] & 0x7FFF) == 0x7FFF).sum().item()
    assert sat > 0, "the boosted gradients should reach the E4M11 finite bound"
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["e4", "fp16"])
def test_gpt2_148_full(pa, mode):
    import torch

    b = _bench()
    w = b.Workload("gpt2-148", mode, torch.device("cuda"), seed=99)
    run = b.step_fn(pa, w, wl.HYPER, None)
    p = w.p.cpu().numpy()
    g = w.g.cpu().numpy()
    s = w.s[0].cpu().numpy().view(np.uint32)
    for t in (1, 2):
        run(t)
        p, s, _ = oracle.step_packed(p, g, s, t, mode=mode, threads=16, **wl.HYPER)
    torch.cuda.synchronize()
    assert_same_bits(w.p.cpu().numpy(), p, f"{mode} p")
    assert_same_bits(w.s[0].cpu().numpy().view(np.uint32), s, f"{mode} state")


def test_blockwise_1e9_sampled(pa):
    import torch

    b = _bench()
    w = b.Workload("blockwise-1e9", "e4", torch.device("cuda"), seed=5)
    n, B = w.n, 2048
    nb = -(-n // B)
    run = b.step_fn(pa, w, wl.HYPER, None)
    q1, q2 = w.q1.cpu().numpy(), w.q2.cpu().numpy()
    rng = np.random.default_rng(3)
    blocks = sorted(set(rng.integers(0, nb - 1, 62).tolist()) | {0, nb - 1})

    def grab(blk):
        a, e = blk * B, min(n, (blk + 1) * B)
        return [w.p[a:e].cpu().numpy(), w.g[a:e].cpu().numpy(), w.m_code[a:e].cpu().numpy(),
                w.m_absmax[blk:blk + 1].cpu().numpy(), w.v_code[a:e].cpu().numpy(),
                w.v_absmax[blk:blk + 1].cpu().numpy()]

    host = {blk: grab(blk) for blk in blocks}
    for t in (1, 2):
        run(t)
        torch.cuda.synchronize()
        for blk in blocks:
            p, g, mc, ma, vc, va = host[blk]
            ob, mc, ma, vc, va, _ = oracle.step_blockwise8(p, g, mc, ma, vc, va, q1, q2, t,
                                                           **wl.HYPER)
            host[blk] = [p, g, mc, ma, vc, va]
            a, e = blk * B, min(n, (blk + 1) * B)
            got = w.p_bf16[a:e].view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ob), f"bf16 block {blk} step {t}"
            assert np.array_equal(w.m_code[a:e].cpu().numpy(), mc)
            assert np.array_equal(w.v_code[a:e].cpu().numpy(), vc)
            assert_same_f32_nan_aware(w.m_absmax[blk:blk + 1].cpu().numpy(), ma)
            assert_same_f32_nan_aware(w.v_absmax[blk:blk + 1].cpu().numpy(), va)
    del w
    torch.cuda.empty_cache()


def test_turbo_124m_sampled(pa):
    """turbo-124m (GPT-2 small's 124,439,808 parameters): three TurboAdam-style
    steps at full size, the bench's launch; 48 sampled slices of eight
    128-value blocks (the first and the short last one included) against the
    oracle's step over each slice, its rounding counters at the tensor's
    element indices (whole blocks are independent given the tensor's scales,
    which every slice takes from the GPU's state before the step)."""
    import torch

    b = _bench()
    w = b.Workload("turbo-124m", "turbo", torch.device("cuda"), seed=11)
    n = w.n
    run = b.step_fn(pa, w, wl.HYPER, None)
    nb = -(-n // 128)
    rng = np.random.default_rng(8)
    starts = sorted(set((rng.integers(0, nb - 8, 46) * 128).tolist()) | {0, (nb - 1) * 128})

    def host_state():
        out = {}
        for k in ("ucode", "umean", "uscal", "vidx", "vend"):
            a = w.st[k].cpu().numpy()
            out[k] = a.view(np.uint16) if a.dtype == np.int16 else a.copy()
        return out

    def cut(st, s0, length):
        return {"ucode": st["ucode"][s0 // 4:(s0 + length + 3) // 4],
                "umean": st["umean"][s0 // 64:(s0 + length + 63) // 64],
                "vidx": st["vidx"][s0 // 2:(s0 + length + 1) // 2],
                "vend": st["vend"][2 * (s0 // 128):2 * ((s0 + length + 127) // 128)]}

    g = w.g.cpu().numpy()
    for t in (1, 2, 3):
        before, p = host_state(), w.p.cpu().numpy()
        run(t)
        torch.cuda.synchronize()
        after, p_gpu = host_state(), w.p.cpu().numpy()
        for s0 in starts:
            length = min(1024, n - s0)
            sl = cut(before, s0, length)
            sl["uscal"] = before["uscal"].copy()
            ps, sts, _ = oracle.turbo_step(p[s0:s0 + length], g[s0:s0 + length], sl, t,
                                           index0=s0, **wl.HYPER)
            assert_same_bits(p_gpu[s0:s0 + length], ps, f"turbo p, step {t}, slice {s0}")
            got = cut(after, s0, length)
            for k in got:
                assert np.array_equal(got[k], sts[k]), (t, s0, k)
