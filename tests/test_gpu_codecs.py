"""GPU codecs against the CPU oracle, bit for bit (pa_encode_state /
pa_decode_state and the FP16 variants, called through the C ABI).

"Packed AdamW Reference" README v1.0.0, "The canonical format": low 16 bits
signed finite E4M11 first moment, high 16 bits unsigned finite E4M12
uncorrected RMS; the FP16-first/FP16-RMS comparison mode.
"""
import numpy as np
import pytest

import oracle
import pins
from gpu_helpers import assert_same_bits, dev, host_f32, host_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import adamw_update_gb300

    return adamw_update_gb300


def _probe_values():
    rng = np.random.default_rng(101)
    x = pins._e4_probe_values(oracle.default(), rng, count=300_000)
    special = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, 65504, 65520, 1e-45,
                        -1e-45, 2.0, -2.0, 1e30, -1e30], np.float32)
    return np.concatenate([x, special]).astype(np.float32)


@pytest.mark.parametrize("mode", ["e4", "fp16"])
def test_decode_every_word_lane(pa, mode):
    import torch

    codes = np.arange(65536, dtype=np.uint32)
    words = (codes << 16) | codes  # every code in both lanes
    m = torch.empty(65536, dtype=torch.float32, device="cuda")
    r = torch.empty_like(m)
    fn = pa.pa_decode_state if mode == "e4" else pa.pa_decode_state_fp16
    fn(dev(words), m, r)
    em, er = oracle.decode_state(words, mode=mode)
    gm, gr = host_f32(m), host_f32(r)
    if mode == "fp16":  # binary16 NaN codes decode to some NaN on both sides
        nan = np.isnan(em)
        assert np.isnan(gm[nan]).all() and np.isnan(gr[nan]).all()
        em, gm, er, gr = em[~nan], gm[~nan], er[~nan], gr[~nan]
    assert_same_bits(gm, em, f"{mode} m lane decode")
    assert_same_bits(gr, er, f"{mode} rms lane decode")


@pytest.mark.parametrize("mode", ["e4", "fp16"])
def test_encode_probe_values(pa, mode):
    import torch

    x = _probe_values()
    rng = np.random.default_rng(7)
    y = rng.permutation(x)
    w = torch.empty(x.size, dtype=torch.int32, device="cuda")
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    fn = pa.pa_encode_state if mode == "e4" else pa.pa_encode_state_fp16
    fn(dev(x), dev(y), w, nonfinite=bad)
    exp, exp_bad = oracle.encode_state(x, y, mode=mode)
    assert_same_bits(host_u32(w), exp, f"{mode} encode")
    assert int(bad.item()) == exp_bad


@pytest.mark.parametrize("mode", ["e4", "fp16"])
def test_roundtrip_all_codes(pa, mode):
    import torch

    codes = np.arange(65536, dtype=np.uint32)
    words = (codes << 16) | codes[::-1]
    if mode == "fp16":  # finite binary16 codes only, RMS lane non-negative
        words = words[((words & 0x7C00) != 0x7C00) & (((words >> 16) & 0x7C00) != 0x7C00)]
    m = torch.empty(words.size, dtype=torch.float32, device="cuda")
    r = torch.empty_like(m)
    w = torch.empty(words.size, dtype=torch.int32, device="cuda")
    dec = pa.pa_decode_state if mode == "e4" else pa.pa_decode_state_fp16
    enc = pa.pa_encode_state if mode == "e4" else pa.pa_encode_state_fp16
    dec(dev(words), m, r)
    enc(m, r, w)
    exp = oracle.encode_state(*oracle.decode_state(words, mode=mode), mode=mode)[0]
    assert_same_bits(host_u32(w), exp, f"{mode} round trip")
    if mode == "e4":  # the E4 RMS lane is unsigned: every high code survives
        assert np.array_equal(host_u32(w) >> 16, words >> 16)


def test_empty_and_errors(pa):
    import torch

    e = torch.empty(0, dtype=torch.float32, device="cuda")
    pa.pa_encode_state(e, e, torch.empty(0, dtype=torch.int32, device="cuda"))
    with pytest.raises(pa.PackedAdamError) as ei:
        pa._check(pa._lib.pa_encode_state(None, None, None, 4, None, None))
    assert ei.value.status == 1


@pytest.mark.parametrize("mode", ["e4", "fp16"])
def test_codecs_at_every_phase_and_size(pa, mode):
    """Views at each 4-byte phase (the vectorised kernels peel a head of up to 3
    elements and code a tail of up to 3 one by one) and arrays whose phases
    differ (the per-element kernels): encode and decode equal the oracle."""
    import torch

    rng = np.random.default_rng(77)
    enc = pa.pa_encode_state if mode == "e4" else pa.pa_encode_state_fp16
    dec = pa.pa_decode_state if mode == "e4" else pa.pa_decode_state_fp16
    for n in (1, 3, 4, 5, 7, 8, 9, 4097, 100_003):
        for phases in ((0, 0, 0), (1, 1, 1), (2, 2, 2), (3, 3, 3), (0, 1, 2), (3, 0, 0)):
            m = rng.normal(0, 1e-3, n).astype(np.float32)
            r = np.abs(rng.normal(0, 1e-3, n)).astype(np.float32)
            bufs = [torch.zeros(n + 8, dtype=dt, device="cuda")
                    for dt in (torch.float32, torch.float32, torch.int32)]
            dm, dr, dw = (b[o:o + n] for b, o in zip(bufs, phases))
            dm.copy_(dev(m))
            dr.copy_(dev(r))
            bad = torch.zeros(1, dtype=torch.int64, device="cuda")
            enc(dm, dr, dw, nonfinite=bad)
            torch.cuda.synchronize()
            ew, _ = oracle.encode_state(m, r, mode=mode)
            assert np.array_equal(host_u32(dw), ew), (n, phases)
            assert int(bad.item()) == 0
            dm.zero_()
            dr.zero_()
            dec(dw, dm, dr)
            torch.cuda.synchronize()
            em, er = oracle.decode_state(ew, mode=mode)
            assert np.array_equal(host_f32(dm).view(np.uint32), em.view(np.uint32)), (n, phases)
            assert np.array_equal(host_f32(dr).view(np.uint32), er.view(np.uint32)), (n, phases)
            assert not any(b[:o].any() or b[o + n:].any() for b, o in zip(bufs, phases)), \
                "write outside the views"
