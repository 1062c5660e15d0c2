"""The graph-replayable packed-E4 step: scalars from a device table of rows
indexed on the device.  Uncaptured calls equal the regular tensor-list step;
a CUDA graph captured once replays as consecutive steps equal to the oracle;
a per-step learning-rate schedule; an index past the table sets the status
word and changes nothing."""
import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
HY = wl.HYPER
SIZES = [3, 4097, 20_000, 1]


def _setup(seed):
    import torch

    rng = np.random.default_rng(seed)
    ps = [rng.normal(0, 0.02, n).astype(np.float32) for n in SIZES]
    gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n in SIZES]
    dp = [torch.from_numpy(p.copy()).cuda() for p in ps]
    dg = [torch.from_numpy(g).cuda() for g in gs]
    ds = [torch.zeros(n, dtype=torch.int32, device="cuda") for n in SIZES]
    return ps, gs, dp, dg, ds


def test_table_step_equals_regular_step():
    import torch

    import adamw_update_gb300 as pa

    ps, gs, dp, dg, ds = _setup(1)
    _, _, dp2, dg2, ds2 = _setup(1)
    rows = torch.empty(10 * 8, dtype=torch.float32, device="cuda")
    pa.pa_hyper_table_fill(rows, 1, 10, **HY)
    index = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in range(1, 6):
        pa.pa_adamw_step_packed_e4_multi_graph(list(zip(dp, dg, ds)), rows, 10, index)
        pa.pa_adamw_step_packed_e4_multi(list(zip(dp2, dg2, ds2)), t, **HY)
    torch.cuda.synchronize()
    assert int(index.item()) == 5
    for a, b, c, d in zip(dp, dp2, ds, ds2):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)) and torch.equal(c, d)


def test_captured_graph_replays_consecutive_steps():
    import torch

    import adamw_update_gb300 as pa

    ps, gs, dp, dg, ds = _setup(2)
    entries = pa.tensor_list(list(zip(dp, dg, ds)))
    rows = torch.empty(16 * 8, dtype=torch.float32, device="cuda")
    sched = [1e-3 * (0.9 ** k) for k in range(16)]
    pa.pa_hyper_table_fill(rows, 1, 16, lr_per_step=sched, beta1=HY["beta1"], beta2=HY["beta2"],
                           eps=HY["eps"], wd=HY["wd"])
    index = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside capture: makes the descriptor table
        pa.pa_adamw_step_packed_e4_multi_graph(entries, rows, 16, index, status)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.pa_adamw_step_packed_e4_multi_graph(entries, rows, 16, index, status)
    for _ in range(4):
        graph.replay()
    torch.cuda.synchronize()
    assert int(index.item()) == 5 and int(status.item()) == 0
    hp = [p.copy() for p in ps]
    hs = [np.zeros(n, np.uint32) for n in SIZES]
    for t in range(1, 6):
        for k in range(len(SIZES)):
            hp[k], hs[k], _ = oracle.step_packed(hp[k], gs[k], hs[k], t, lr=sched[t - 1],
                                                 beta1=HY["beta1"], beta2=HY["beta2"],
                                                 eps=HY["eps"], wd=HY["wd"])
    for k in range(len(SIZES)):
        assert np.array_equal(dp[k].cpu().numpy().view(np.uint32), hp[k].view(np.uint32))
        assert np.array_equal(ds[k].cpu().numpy().view(np.uint32), hs[k])


def test_index_past_the_table_changes_nothing():
    import torch

    import adamw_update_gb300 as pa

    _, _, dp, dg, ds = _setup(3)
    rows = torch.empty(2 * 8, dtype=torch.float32, device="cuda")
    pa.pa_hyper_table_fill(rows, 1, 2, **HY)
    index = torch.full((1,), 2, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = [p.clone() for p in dp]
    pa.pa_adamw_step_packed_e4_multi_graph(list(zip(dp, dg, ds)), rows, 2, index, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1 and int(index.item()) == 3
    for a, b, s in zip(dp, before, ds):
        assert torch.equal(a, b) and not s.any()


def test_captured_graph_survives_many_other_lists():
    """A captured launch holds its list's descriptor table: stepping more other
    lists than the table cache keeps (64) between replays must not free it, so
    later replays still step the captured tensors, bit for bit as the oracle."""
    import torch

    import adamw_update_gb300 as pa

    ps, gs, dp, dg, ds = _setup(4)
    entries = pa.tensor_list(list(zip(dp, dg, ds)))
    rows = torch.empty(8 * 8, dtype=torch.float32, device="cuda")
    pa.pa_hyper_table_fill(rows, 1, 8, **HY)
    index = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pa.pa_adamw_step_packed_e4_multi_graph(entries, rows, 8, index, status)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.pa_adamw_step_packed_e4_multi_graph(entries, rows, 8, index, status)
    graph.replay()
    # 70 other two-tensor lists, each a distinct table
    others = []
    for k in range(70):
        a = [torch.zeros(64 + k, device="cuda") for _ in range(2)]
        b = [torch.zeros(64 + k, device="cuda") for _ in range(2)]
        c = [torch.zeros(64 + k, dtype=torch.int32, device="cuda") for _ in range(2)]
        others.append((a, b, c))
        pa.pa_adamw_step_packed_e4_multi(list(zip(a, b, c)), 1, **HY)
    torch.cuda.synchronize()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert int(index.item()) == 4 and int(status.item()) == 0
    hp = [p.copy() for p in ps]
    hs = [np.zeros(n, np.uint32) for n in SIZES]
    for t in range(1, 5):
        for k in range(len(SIZES)):
            hp[k], hs[k], _ = oracle.step_packed(hp[k], gs[k], hs[k], t, **HY)
    for k in range(len(SIZES)):
        assert np.array_equal(dp[k].cpu().numpy().view(np.uint32), hp[k].view(np.uint32))
        assert np.array_equal(ds[k].cpu().numpy().view(np.uint32), hs[k])
