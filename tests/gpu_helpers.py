"""Helpers shared by the GPU parity tests: device copies and bitwise checks."""
from __future__ import annotations

import numpy as np


def dev(a, dtype=None):
    """numpy -> contiguous CUDA tensor (uint32 arrays travel as int32 bits)."""
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    t = torch.from_numpy(a.copy()).cuda()
    return t if dtype is None else t.to(dtype)


def host_u32(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def host_f32(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.float32, copy=False)


def assert_same_bits(got, exp, what=""):
    got = np.ascontiguousarray(got).view(np.uint32)
    exp = np.ascontiguousarray(exp).view(np.uint32)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {got.size} differ; first {bad[:6]} "
                           f"got {got[bad[:6]]} expected {exp[bad[:6]]}")


def assert_same_f32_nan_aware(got, exp, what=""):
    """Bitwise equal, except that any NaN matches any NaN."""
    got = np.ascontiguousarray(got, np.float32)
    exp = np.ascontiguousarray(exp, np.float32)
    nan = np.isnan(got) & np.isnan(exp)
    g = got.view(np.uint32)[~nan]
    e = exp.view(np.uint32)[~nan]
    bad = np.nonzero(g != e)[0]
    assert bad.size == 0, f"{what}: {bad.size} differ; got {g[bad[:6]]} expected {e[bad[:6]]}"
