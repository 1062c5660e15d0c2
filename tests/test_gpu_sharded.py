"""The ZeRO-1 sharded step on one GPU through NCCL (world size 1: the
reduce-scatter and all-gather are the identity, the shard is the whole flat
buffer): the library's step inside the sharded wrapper equals the CPU oracle,
bit for bit, over three steps, in each mode.  The exchanges between two ranks
are covered on the CPU by test_sharded_gloo.py."""
import socket

import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
N = 50_003


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module")
def nccl_group():
    import torch.distributed as dist

    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1)
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["e4", "fp16", "fp32"])
def test_sharded_step_on_one_gpu_equals_the_oracle(nccl_group, mode):
    import torch

    from adamw_update_gb300 import sharded

    hy = wl.HYPER
    L = sharded.padded_length(N, 1)
    flat = torch.zeros(L, dtype=torch.float32, device="cuda")
    p = wl.normal_np(N, 0.02, 3)
    sharded.flatten_into([torch.from_numpy(p).cuda()], flat)
    opt = sharded.ShardedPackedAdamW(flat, mode=mode, lr=hy["lr"],
                                     betas=(hy["beta1"], hy["beta2"]), eps=hy["eps"],
                                     weight_decay=hy["wd"], average=True)
    st = [np.zeros(N, np.float32), np.zeros(N, np.float32)] if mode == "fp32" \
        else [np.zeros(N, np.uint32)]
    gflat = torch.zeros(L, dtype=torch.float32, device="cuda")
    for t in range(1, 4):
        g = wl.normal_np(N, 1e-3, 100 + t)
        gflat[:N] = torch.from_numpy(g).cuda()
        opt.step(gflat)
        if mode == "fp32":
            p, st[0], st[1], _ = oracle.step_fp32(p, g, st[0], st[1], t, **hy)
        else:
            p, st[0], _ = oracle.step_packed(p, g, st[0], t, mode=mode, **hy)
    torch.cuda.synchronize()
    got = flat.cpu().numpy()
    assert np.array_equal(got[:N].view(np.uint32), p.view(np.uint32))
    assert not got[N:].any()
    for s_dev, s_exp in zip(opt.state, st):
        assert np.array_equal(s_dev[:N].cpu().numpy().view(np.uint32), s_exp.view(np.uint32))
    assert int(opt.nonfinite.item()) == 0
