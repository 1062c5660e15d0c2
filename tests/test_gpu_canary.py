"""Out-of-bounds writes, checked without a sanitizer: every buffer handed to
the library is a view in the middle of a larger allocation whose guard bands
(before and after, at least 4 KiB) hold a fixed byte pattern; after the calls
the pattern must be intact.  Sizes are odd and tiny, views start at every
4-byte phase, tensor lists mix phases."""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
GUARD = 4096  # bytes on each side
PATTERN = 0xA5


class Guarded:
    """A view of `n` elements of `dtype`, `offset` elements into the body,
    with canary bytes around it."""

    def __init__(self, n, dtype, offset=0, fill=None):
        import torch

        self.dtype = dtype
        es = torch.empty(0, dtype=dtype).element_size()
        self.lo = GUARD + offset * es
        self.nbytes = n * es
        total = self.lo + self.nbytes + GUARD
        self.raw = torch.full((total,), PATTERN, dtype=torch.uint8, device="cuda")
        self.view = self.raw[self.lo:self.lo + self.nbytes].view(dtype)
        if fill is not None:
            self.view.copy_(fill)

    def intact(self):
        r = self.raw.cpu().numpy()
        return bool((r[: self.lo] == PATTERN).all() and (r[self.lo + self.nbytes:] == PATTERN).all())


def _f32(n, seed, std):
    import torch

    return torch.from_numpy(np.random.default_rng(seed).normal(0, std, n).astype(np.float32))


@pytest.mark.parametrize("n", [1, 2, 3, 5, 17, 4095, 4097, 6143, 6145, 9001, 12291])
@pytest.mark.parametrize("off", [0, 1, 2, 3])
def test_single_steps_and_codecs_stay_in_bounds(n, off):
    import torch

    import adamw_update_gb300 as pa

    p = Guarded(n, torch.float32, off, _f32(n, 1, 0.02))
    g = Guarded(n, torch.float32, off, _f32(n, 2, 1e-3))
    gb = Guarded(n, torch.bfloat16, off, _f32(n, 3, 1e-3).to(torch.bfloat16))
    s = Guarded(n, torch.int32, off)
    s.view.zero_()
    m = Guarded(n, torch.float32, (off + 1) % 4, _f32(n, 4, 1e-4))
    v = Guarded(n, torch.float32, off, _f32(n, 5, 1e-4).abs())
    cnt = Guarded(1, torch.int64)
    cnt.view.zero_()
    pa.pa_adamw_step_packed_e4(p.view, g.view, s.view, 1, nonfinite=cnt.view, **wl.HYPER)
    pa.pa_adamw_step_packed_fp16(p.view, g.view, s.view, 2, **wl.HYPER)
    pa.pa_adamw_step_fp32(p.view, g.view, m.view, v.view, 3, **wl.HYPER)
    pa.pa_adamw_step_packed_e4_bf16g(p.view, gb.view, s.view, 4, **wl.HYPER)
    pa.pa_adamw_step_packed_e4_multi([(p.view, g.view, s.view)], 5, **wl.HYPER)
    pa.pa_adamw_step_fp32_multi([(p.view, g.view, m.view, v.view)], 6, **wl.HYPER)
    w = Guarded(n, torch.int32, off)
    pa.pa_encode_state(m.view, v.view, w.view)
    pa.pa_decode_state(w.view, m.view, v.view)
    pa.pa_encode_state_fp16(m.view, v.view, w.view)
    pa.pa_decode_state_fp16(w.view, m.view, v.view)
    torch.cuda.synchronize()
    for b in (p, g, gb, s, m, v, cnt, w):
        assert b.intact()


def test_tensor_lists_stay_in_bounds():
    import torch

    import adamw_update_gb300 as pa

    sizes = [1, 0, 3, 4096, 5, 10_007, 2]
    bufs = []
    for k, n in enumerate(sizes):
        bufs.append((Guarded(n, torch.float32, k % 4, _f32(n, k, 0.02)),
                     Guarded(n, torch.float32, (k + 1) % 4, _f32(n, k + 10, 1e-3)),
                     Guarded(n, torch.int32, k % 4)))
    for _, _, s in bufs:
        s.view.zero_()
    entries = [(p.view, g.view, s.view) for p, g, s in bufs]
    for t in range(1, 4):
        pa.pa_adamw_step_packed_e4_multi(entries, t, **wl.HYPER)
        pa.pa_adamw_step_packed_fp16_multi(entries, t, **wl.HYPER)
        pa.pa_adamw_step_packed_e4_multi_noalloc(entries, t, **wl.HYPER)
    torch.cuda.synchronize()
    for trio in bufs:
        assert all(b.intact() for b in trio)


@pytest.mark.parametrize("n", [1, 5, 2047, 2048, 2049, 3 * 2048 + 7])
def test_blockwise_stays_in_bounds(n):
    import torch

    import adamw_update_gb300 as pa

    nb = -(-n // 2048)
    q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
    p = Guarded(n, torch.float32, 0, _f32(n, 1, 0.02))
    g = Guarded(n, torch.float32, 0, _f32(n, 2, 1e-3))
    out = Guarded(n, torch.bfloat16, 0)
    mc = Guarded(n, torch.uint8, 0)
    vc = Guarded(n, torch.uint8, 0)
    mc.view.fill_(wl.nearest_zero_code(q1))
    vc.view.fill_(wl.nearest_zero_code(q2))
    ma = Guarded(nb, torch.float32, 1)
    va = Guarded(nb, torch.float32, 3)
    ma.view.zero_()
    va.view.zero_()
    d1 = Guarded(256, torch.float32, 0, torch.from_numpy(q1))
    d2 = Guarded(256, torch.float32, 0, torch.from_numpy(q2))
    for t in (1, 2):
        pa.pa_adamw_step_blockwise8(p.view, g.view, out.view, mc.view, ma.view, vc.view, va.view,
                                    d1.view, d2.view, t)
    torch.cuda.synchronize()
    for b in (p, g, out, mc, vc, ma, va, d1, d2):
        assert b.intact()


def test_host_step_workspace_stays_in_bounds():
    import torch

    import adamw_update_gb300 as pa

    n = 200_001
    ws = Guarded(3 * 12 * 65536, torch.uint8, 0)
    hp = _f32(n, 1, 0.02).pin_memory()
    hg = _f32(n, 2, 1e-3).pin_memory()
    hs = torch.zeros(n, dtype=torch.int32).pin_memory()
    pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws.view, 1, **wl.HYPER)
    torch.cuda.current_stream().synchronize()
    assert ws.intact()
