"""Seeded synthetic inputs for the packed-state AdamW update.

Shared by the tests, the smoke check and bench.py, and the only thing the
oracle and the CUDA path have in common: they are handed the same bytes.  This
module holds none of the update's arithmetic -- only shapes, random
distributions and the ascending 256-entry maps that the blockwise mode takes
as inputs.

The workloads (synthetic stand-ins; the pages' token tapes are not available):

  single-4096    one FP32 tensor of 4,096 parameters, p ~ N(0, 0.02),
                 g ~ N(0, 1e-3) drawn fresh each step, zero state.
  gpt-52         the 52-tensor list of the pages' learned-position GPT shapes
                 (token embedding 12096x256, position 1024x256, 8 layers of
                 qkv 256x768+768, proj 256x256+256, fc 256x1024+1024,
                 out 1024x256+256 and two LayerNorms of 256+256, final
                 LayerNorm 256+256); each bias is folded into its weight.
  gpt2-148       GPT-2-small shapes (vocab 50257, d 768, 12 layers, context
                 1024): 148 tensors, biases separate; per tensor
                 g ~ N(0, s) with log10 s ~ U(-5, -1) and 1 % exact zeros.
  flat-7e9       one flat tensor of 7e9 parameters; g = 1e-3 * t(df=3) with a
                 1e-4 fraction of entries scaled by 1e4.
  blockwise-1e9  1e9 parameters for the 8-bit blockwise mode, g ~ N(0, 1e-3),
                 codes start at the map entry nearest 0 and absmax at 0.
  turbo-124m     the TurboAdam-style step on one tensor of GPT-2 small's
                 124,439,808 parameters (the TurboAdam page's language-model
                 runs are GPT-2 124M), g ~ N(0, 1e-3) with half the entries
                 scaled by 10, zero state.
"""
from __future__ import annotations

import math

import numpy as np

GPT52_SHAPES = (
    [("tok_emb", 12096 * 256), ("pos_emb", 1024 * 256)]
    + [
        (f"h{i}.{name}", size)
        for i in range(8)
        for name, size in (
            ("qkv", 256 * 768 + 768),
            ("proj", 256 * 256 + 256),
            ("fc", 256 * 1024 + 1024),
            ("out", 1024 * 256 + 256),
            ("ln1", 256 + 256),
            ("ln2", 256 + 256),
        )
    ]
    + [("lnf.w", 256), ("lnf.b", 256)]
)

GPT2_148_SHAPES = (
    [("wte", 50257 * 768), ("wpe", 1024 * 768)]
    + [
        (f"h{i}.{name}", size)
        for i in range(12)
        for name, size in (
            ("ln_1.w", 768), ("ln_1.b", 768),
            ("attn.c_attn.w", 768 * 2304), ("attn.c_attn.b", 2304),
            ("attn.c_proj.w", 768 * 768), ("attn.c_proj.b", 768),
            ("ln_2.w", 768), ("ln_2.b", 768),
            ("mlp.c_fc.w", 768 * 3072), ("mlp.c_fc.b", 3072),
            ("mlp.c_proj.w", 3072 * 768), ("mlp.c_proj.b", 768),
        )
    ]
    + [("ln_f.w", 768), ("ln_f.b", 768)]
)

WORKLOADS = {
    "single-4096": dict(n=4096, steps=10),
    "gpt-52": dict(n=sum(s for _, s in GPT52_SHAPES), steps=100),
    "gpt2-148": dict(n=sum(s for _, s in GPT2_148_SHAPES), steps=50),
    "flat-7e9": dict(n=7_000_000_000, steps=20),
    "blockwise-1e9": dict(n=1_000_000_000, steps=1),
    "turbo-124m": dict(n=sum(s for _, s in GPT2_148_SHAPES), steps=20),
}

HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)

_CHUNK = 1 << 26


def _gen(seed: int, stream: int, chunk: int, device):
    import torch

    g = torch.Generator(device=device)
    # distinct, reproducible seed per (seed, stream, chunk)
    g.manual_seed((seed * 1_000_003 + stream * 7_919 + chunk * 104_729) % (1 << 62))
    return g


def fill_normal_(t, std: float, seed: int, stream: int = 0):
    """Fill a 1-D FP32 tensor with N(0, std^2), chunk by chunk."""
    import torch

    n = t.numel()
    for k, lo in enumerate(range(0, n, _CHUNK)):
        hi = min(n, lo + _CHUNK)
        g = _gen(seed, stream, k, t.device)
        t[lo:hi].copy_(torch.randn(hi - lo, generator=g, device=t.device, dtype=torch.float32) * std)
    return t


def fill_student_t_saturating_(t, seed: int, stream: int = 1, scale: float = 1e-3,
                               frac: float = 1e-4, boost: float = 1e4):
    """g = scale * t(df=3), with a `frac` share of entries multiplied by `boost`."""
    import torch

    n = t.numel()
    for k, lo in enumerate(range(0, n, _CHUNK)):
        hi = min(n, lo + _CHUNK)
        m = hi - lo
        g = _gen(seed, stream, k, t.device)
        z = torch.randn(m, generator=g, device=t.device, dtype=torch.float32)
        chi = torch.randn(3, m, generator=g, device=t.device, dtype=torch.float32).square().sum(0)
        tt = z / torch.sqrt(chi / 3.0)
        u = torch.rand(m, generator=g, device=t.device, dtype=torch.float32)
        tt = torch.where(u < frac, tt * boost, tt)
        t[lo:hi].copy_(tt * scale)
    return t


def fill_gpt2_grads_(flat, sizes, seed: int, stream: int = 2):
    """Per-tensor g ~ N(0, s), log10 s ~ U(-5, -1), 1 % of entries exactly zero."""
    import torch

    rng = np.random.default_rng(seed + 17)
    off = 0
    for k, n in enumerate(sizes):
        s = float(10.0 ** rng.uniform(-5.0, -1.0))
        seg = flat[off:off + n]
        g = _gen(seed, stream, k, flat.device)
        x = torch.randn(n, generator=g, device=flat.device, dtype=torch.float32) * s
        keep = torch.rand(n, generator=g, device=flat.device, dtype=torch.float32) >= 0.01
        seg.copy_(torch.where(keep, x, torch.zeros_like(x)))
        off += n
    return flat


# ---- ascending 256-entry maps for the blockwise mode (inputs, not method) ----

def _f32_sorted_unique(vals):
    a = np.unique(np.asarray(vals, dtype=np.float64).astype(np.float32))
    assert a.size == 256, a.size
    assert np.all(np.diff(a) > 0)
    return a


def dynamic_qmap_signed() -> np.ndarray:
    """Signed log-and-linear map in [-1, 1]: per decade 10^-d (d = 0..6), the
    fractions 0.15, 0.20, ..., 1.00 of it; 0; the smallest magnitudes 1e-7 and
    5e-8 (the latter positive only), so that 256 entries result."""
    pos = [10.0 ** -d * (0.10 + 0.05 * k) for d in range(7) for k in range(1, 19)]
    pos += [1e-7]
    vals = [0.0] + pos + [-x for x in pos] + [5e-8]
    return _f32_sorted_unique(vals)


def dynamic_qmap_unsigned() -> np.ndarray:
    """Unsigned log-and-linear map in [0, 1]: per decade 10^-d (d = 0..6), the
    fractions 0.125, 0.150, ..., 1.000 of it; 0; and 1e-7, 5e-8, 2.5e-8."""
    pos = [10.0 ** -d * (0.100 + 0.025 * k) for d in range(7) for k in range(1, 37)]
    vals = [0.0] + pos + [1e-7, 5e-8, 2.5e-8]
    return _f32_sorted_unique(vals)


def linear_qmap_signed() -> np.ndarray:
    """Uniform map: -1 + 2 i / 255, i = 0 .. 255."""
    return (-1.0 + 2.0 * np.arange(256, dtype=np.float64) / 255.0).astype(np.float32)


def linear_qmap_unsigned() -> np.ndarray:
    """Uniform map: i / 255, i = 0 .. 255."""
    return (np.arange(256, dtype=np.float64) / 255.0).astype(np.float32)


def random_qmap(seed: int, signed: bool) -> np.ndarray:
    """A random strictly ascending map with exact endpoints (0 or -1, and 1)."""
    rng = np.random.default_rng(seed)
    lo = -1.0 if signed else 0.0
    while True:
        inner = rng.uniform(lo, 1.0, 254)
        a = np.unique(np.concatenate([[lo, 1.0], inner]).astype(np.float32))
        if a.size == 256:
            return a


def nearest_zero_code(qmap: np.ndarray) -> int:
    """Index of the map entry of smallest magnitude (the initial state code)."""
    return int(np.argmin(np.abs(qmap.astype(np.float64))))


def normal_np(n: int, std: float, seed: int) -> np.ndarray:
    """Host-side N(0, std^2) FP32 sample (small cases)."""
    return (np.random.default_rng(seed).standard_normal(n) * std).astype(np.float32)


def blocks(n: int, block: int = 2048) -> int:
    return math.ceil(n / block)


def fill_turbo_grads_(t, seed: int, stream: int = 3):
    """g ~ N(0, 1e-3), half the entries (a seeded coin) scaled by 10."""
    import torch

    n = t.numel()
    for k, lo in enumerate(range(0, n, _CHUNK)):
        hi = min(n, lo + _CHUNK)
        g = _gen(seed, stream, k, t.device)
        x = torch.randn(hi - lo, generator=g, device=t.device, dtype=torch.float32) * 1e-3
        big = torch.rand(hi - lo, generator=g, device=t.device, dtype=torch.float32) < 0.5
        t[lo:hi].copy_(torch.where(big, x * 10.0, x))
    return t
