"""The packed-E4 step over host-resident tensors (pa_adamw_step_packed_e4_host),
bit for bit equal to the oracle: pinned tensors (the kernel reads and writes
them in place over the host link), pageable or mixed ones (streamed through a
small device workspace in many chunks with a ragged last chunk), views into
pinned buffers at odd offsets, two calls in a row ("Packed AdamW Reference" README, "The canonical format":
the 4-byte state word is what travels between host and device)."""
import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
HY = wl.HYPER


@pytest.mark.parametrize("pinned", [True, False])
def test_host_step_matches_oracle(pinned):
    import torch

    import adamw_update_gb300 as pa

    n = 1_000_003  # 16 chunks of 65,536 with a ragged tail
    rng = np.random.default_rng(5)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = np.zeros(n, np.uint32)
    hp = torch.from_numpy(p.copy())
    hs = torch.zeros(n, dtype=torch.int32)
    if pinned:
        hp, hs = hp.pin_memory(), hs.pin_memory()
    ws = torch.empty(3 * 12 * 65536, dtype=torch.uint8, device="cuda")
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in (1, 2):
        g = (1e-3 * rng.standard_t(3, n)).astype(np.float32)
        hg = torch.from_numpy(g)
        if pinned:
            hg = hg.pin_memory()
        pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws, t, nonfinite=bad, **HY)
        torch.cuda.current_stream().synchronize()
        p, st, _ = oracle.step_packed(p, g, st, t, **HY)
        assert np.array_equal(hp.numpy().view(np.uint32), p.view(np.uint32)), f"p, call {t}"
        assert np.array_equal(hs.numpy().view(np.uint32), st), f"state, call {t}"
    assert int(bad.item()) == 0


def test_host_step_small_tensor_and_errors():
    import torch

    import adamw_update_gb300 as pa

    n = 1000
    rng = np.random.default_rng(6)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    hp, hg = torch.from_numpy(p.copy()), torch.from_numpy(g)
    hs = torch.zeros(n, dtype=torch.int32)
    ws = torch.empty(3 * 12 * 65536 + 7, dtype=torch.uint8, device="cuda")
    pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws, 1, **HY)
    torch.cuda.current_stream().synchronize()
    ep, es, _ = oracle.step_packed(p, g, np.zeros(n, np.uint32), 1, **HY)
    assert np.array_equal(hp.numpy().view(np.uint32), ep.view(np.uint32))
    assert np.array_equal(hs.numpy().view(np.uint32), es)
    with pytest.raises(pa.PackedAdamError) as e:
        pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws[: 3 * 12 * 65536 - 1], 2, **HY)
    assert e.value.status == 2
    with pytest.raises(pa.PackedAdamError) as e:
        pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws[1:], 2, **HY)
    assert e.value.status == 3


@pytest.mark.parametrize("case", ["mixed", "offset_views"])
def test_host_step_in_place_and_mixed(case):
    """offset_views: pinned buffers, views starting at 4-byte offsets (in
    place, 4-byte path); mixed: pinned p and state with a pageable gradient
    (streamed through the workspace)."""
    import torch

    import adamw_update_gb300 as pa

    n = 300_007
    rng = np.random.default_rng(7)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    st = rng.integers(0, 1 << 31, n).astype(np.uint32)
    bp = torch.zeros(n + 4, dtype=torch.float32).pin_memory()
    bs = torch.zeros(n + 4, dtype=torch.int32).pin_memory()
    bg = torch.zeros(n + 4, dtype=torch.float32).pin_memory()
    o = (1, 3, 2) if case == "offset_views" else (0, 0, 0)
    hp, hs = bp[o[0]:o[0] + n], bs[o[1]:o[1] + n]
    hp.copy_(torch.from_numpy(p))
    hs.copy_(torch.from_numpy(st.view(np.int32)))
    ws = torch.empty(3 * 12 * 65536, dtype=torch.uint8, device="cuda")
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in (1, 2):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        if case == "offset_views":
            hg = bg[o[2]:o[2] + n]
            hg.copy_(torch.from_numpy(g))
        else:
            hg = torch.from_numpy(g)
        pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws, t, nonfinite=bad, **HY)
        torch.cuda.current_stream().synchronize()
        p, st, _ = oracle.step_packed(p, g, st, t, **HY)
        assert np.array_equal(hp.numpy().view(np.uint32), p.view(np.uint32)), f"p, call {t}"
        assert np.array_equal(hs.numpy().view(np.uint32), st), f"state, call {t}"
    assert int(bad.item()) == 0
