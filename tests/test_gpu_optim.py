"""PackedAdamW (torch.optim.Optimizer over the tensor-list steps) on the GPU:
bit-exact against the oracle tensor by tensor, exact resume from a checkpoint,
the one-word state ledger and the non-finite count ("Packed AdamW Reference"
README v1.0.0: reusable dense optimizer; the smoke check's finite loss, zero
non-finite count, one-word state ledger and checkpoint round trip)."""
import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
HY = wl.HYPER
SIZES = [5, 4097, 300, 70_001, 1]


def _params(seed):
    import torch

    rng = np.random.default_rng(seed)
    return [torch.nn.Parameter(torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).cuda())
            for n in SIZES]


def _grads(rng):
    return [rng.normal(0, 1e-3, n).astype(np.float32) for n in SIZES]


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_optimizer_matches_oracle(mode):
    import torch

    from adamw_update_gb300.optim import PackedAdamW

    params = _params(1)
    opt = PackedAdamW(params, lr=HY["lr"], betas=(HY["beta1"], HY["beta2"]), eps=HY["eps"],
                      weight_decay=HY["wd"], mode=mode)
    host = [p.detach().cpu().numpy().copy() for p in params]
    st = [[np.zeros(n, np.float32), np.zeros(n, np.float32)] if mode == "fp32"
          else [np.zeros(n, np.uint32)] for n in SIZES]
    rng = np.random.default_rng(2)
    for t in range(1, 6):
        gs = _grads(rng)
        for p, g in zip(params, gs):
            p.grad = torch.from_numpy(g).cuda()
        opt.step()
        for k, g in enumerate(gs):
            if mode == "fp32":
                host[k], st[k][0], st[k][1], _ = oracle.step_fp32(host[k], g, *st[k], t, **HY)
            else:
                host[k], st[k][0], _ = oracle.step_packed(host[k], g, st[k][0], t, mode=mode, **HY)
    torch.cuda.synchronize()
    for k, p in enumerate(params):
        assert np.array_equal(p.detach().cpu().numpy().view(np.uint32), host[k].view(np.uint32))
        s = opt.state[p]
        if mode == "fp32":
            assert np.array_equal(s["exp_avg"].cpu().numpy().view(np.uint32), st[k][0].view(np.uint32))
            assert np.array_equal(s["exp_avg_sq"].cpu().numpy().view(np.uint32), st[k][1].view(np.uint32))
        else:
            assert np.array_equal(s["packed"].cpu().numpy().view(np.uint32), st[k][0])
    assert opt.param_groups[0]["step"] == 5


@pytest.mark.parametrize("mode", ["e4", "fp32"])
def test_checkpoint_resume_is_exact(tmp_path, mode):
    import torch

    from adamw_update_gb300.optim import PackedAdamW, load_checkpoint, save_checkpoint

    def run(params, opt, grads):
        for gs in grads:
            for p, g in zip(params, gs):
                p.grad = torch.from_numpy(g).cuda()
            opt.step()
        torch.cuda.synchronize()

    rng = np.random.default_rng(3)
    grads = [_grads(rng) for _ in range(6)]
    params = _params(4)
    opt = PackedAdamW(params, mode=mode, weight_decay=0.01)
    run(params, opt, grads[:3])
    path = str(tmp_path / "latest.pt")
    save_checkpoint(path, params, opt, extra={"update": 3})
    run(params, opt, grads[3:])
    want = [p.detach().clone() for p in params]
    want_state = [{k: v.clone() for k, v in opt.state[p].items()} for p in params]

    params2 = _params(99)  # different values: all must come from the checkpoint
    opt2 = PackedAdamW(params2, mode=mode, weight_decay=0.01)
    assert load_checkpoint(path, params2, opt2) == {"update": 3}
    assert opt2.param_groups[0]["step"] == 3
    run(params2, opt2, grads[3:])
    for p, w, p2, ws in zip(params, want, params2, want_state):
        assert torch.equal(p2.detach().view(torch.int32), w.view(torch.int32))
        for k, v in ws.items():
            assert torch.equal(opt2.state[p2][k].view(torch.int32), v.view(torch.int32)), k


def test_smoke_contract_tiny_model(tmp_path):
    """A tiny MLP trained 30 updates on synthetic data: finite loss, zero
    non-finite count, one 4-byte state word per parameter, and a checkpoint
    round trip."""
    import torch

    from adamw_update_gb300.optim import PackedAdamW, load_checkpoint, save_checkpoint

    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(64, 128), torch.nn.GELU(),
                                torch.nn.Linear(128, 10)).cuda()
    opt = PackedAdamW(model.parameters(), lr=3e-3, weight_decay=0.01)
    x = torch.randn(256, 64, device="cuda")
    y = torch.randint(0, 10, (256,), device="cuda")
    losses = []
    for _ in range(30):
        opt.zero_grad(set_to_none=False)
        loss = torch.nn.functional.cross_entropy(model(x), y)
        loss.backward()
        opt.step()
        losses.append(loss.item())
    assert all(np.isfinite(losses)) and losses[-1] < losses[0]
    assert opt.nonfinite_count() == 0
    nparams = sum(p.numel() for p in model.parameters())
    assert opt.state_bytes() == 4 * nparams
    path = str(tmp_path / "smoke.pt")
    save_checkpoint(path, list(model.parameters()), opt)
    model2 = torch.nn.Sequential(torch.nn.Linear(64, 128), torch.nn.GELU(),
                                 torch.nn.Linear(128, 10)).cuda()
    opt2 = PackedAdamW(model2.parameters(), lr=3e-3, weight_decay=0.01)
    load_checkpoint(path, list(model2.parameters()), opt2)
    for a, b in zip(model.parameters(), model2.parameters()):
        assert torch.equal(a, b)
    for a, b in zip(model.parameters(), model2.parameters()):
        assert torch.equal(opt.state[a]["packed"], opt2.state[b]["packed"])


def test_nonfinite_gradient_is_counted():
    import torch

    from adamw_update_gb300.optim import PackedAdamW

    params = _params(5)
    opt = PackedAdamW(params)
    for p in params:
        p.grad = torch.zeros_like(p)
    params[1].grad[7] = float("nan")
    opt.step()
    assert opt.nonfinite_count() == 1
