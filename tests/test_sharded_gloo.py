"""The ZeRO-1 sharded step (adamw_update_gb300.sharded) on two CPU ranks over
gloo: reduce-scatter of the gradients, each rank's shard stepped, all-gather of
the parameters.  Each rank's step function is the CPU oracle, handed in by
this test (the product never imports the oracle), so what is checked here is
the sharding and the exchanges: after three steps every rank's parameters and
the concatenated state shards equal, bit for bit, the unsharded oracle step
fed with the summed gradients.  Two ranks make the sum order irrelevant
(a + b = b + a exactly in IEEE arithmetic)."""
import os
import socket

import numpy as np
import pytest

N = 10_007  # not a multiple of the shard alignment: the flat buffer is padded
STEPS = 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grads(rank, step, n):
    return np.random.default_rng(1000 * rank + step).normal(0, 1e-3, n).astype(np.float32)


def _oracle_step(mode):
    import torch

    import oracle

    def step(p, g, state, t, hyper, nonfinite):
        if mode == "fp32":
            pn, mn, vn, bad = oracle.step_fp32(p.numpy(), g.numpy(), state[0].numpy(),
                                               state[1].numpy(), t, **hyper)
            state[0].copy_(torch.from_numpy(mn))
            state[1].copy_(torch.from_numpy(vn))
        else:
            pn, sn, bad = oracle.step_packed(p.numpy(), g.numpy(),
                                             state[0].numpy().view(np.uint32), t, mode=mode,
                                             **hyper)
            state[0].copy_(torch.from_numpy(sn.view(np.int32)))
        p.copy_(torch.from_numpy(pn))
        nonfinite += int(bad)
    return step


def _rank(rank, world, port, mode, out):
    import sys

    sys.path[:0] = [os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    os.path.dirname(os.path.abspath(__file__))]
    import torch
    import torch.distributed as dist

    from adamw_update_gb300 import sharded

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        L = sharded.padded_length(N, world)
        flat = torch.zeros(L, dtype=torch.float32)
        p0 = np.random.default_rng(7).normal(0, 0.02, N).astype(np.float32)
        sharded.flatten_into([torch.from_numpy(p0)], flat)
        opt = sharded.ShardedPackedAdamW(flat, mode=mode, lr=1e-3, betas=(0.9, 0.999),
                                         eps=1e-8, weight_decay=0.01, average=False,
                                         step_fn=_oracle_step(mode))
        gflat = torch.zeros(L, dtype=torch.float32)
        for t in range(1, STEPS + 1):
            gflat[:N] = torch.from_numpy(_grads(rank, t, N))
            opt.step(gflat)
        states = []
        for s in opt.state:
            full = torch.zeros(L, dtype=s.dtype)
            dist.all_gather_into_tensor(full, s)
            states.append(full.numpy())
        np.save(os.path.join(out, f"p{rank}.npy"), flat.numpy())
        for k, s in enumerate(states):
            np.save(os.path.join(out, f"s{rank}_{k}.npy"), s)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["e4", "fp32"])
def test_sharded_step_equals_the_unsharded_step(mode, tmp_path, built_package):
    import multiprocessing as mp

    import oracle

    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, mode, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"

    hy = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
    p = np.random.default_rng(7).normal(0, 0.02, N).astype(np.float32)
    if mode == "fp32":
        st = [np.zeros(N, np.float32), np.zeros(N, np.float32)]
    else:
        st = [np.zeros(N, np.uint32)]
    for t in range(1, STEPS + 1):
        g = _grads(0, t, N) + _grads(1, t, N)
        if mode == "fp32":
            p, st[0], st[1], _ = oracle.step_fp32(p, g, st[0], st[1], t, **hy)
        else:
            p, st[0], _ = oracle.step_packed(p, g, st[0], t, mode=mode, **hy)
    for r in range(world):
        got = np.load(tmp_path / f"p{r}.npy")
        assert np.array_equal(got[:N].view(np.uint32), p.view(np.uint32)), f"rank {r} params"
        assert not got[N:].any(), "padding moved"
        for k, s in enumerate(st):
            gs = np.load(tmp_path / f"s{r}_{k}.npy")
            assert np.array_equal(gs[:N].view(np.uint32), s.view(np.uint32)), f"state {k}"
            assert not gs[N:].view(np.uint32).any()


def test_padded_length_gives_equal_aligned_shards(built_package):
    from adamw_update_gb300 import shard_bounds, sharded

    for n in (1, 3, 4, 10_007, 1 << 20):
        for world in (1, 2, 3, 8):
            L = sharded.padded_length(n, world)
            assert L >= n and L % (4 * world) == 0
            assert L - n < 4 * world  # no more padding than alignment needs
            shards = [shard_bounds(L, world, r) for r in range(world)]
            assert all(hi - lo == L // world for lo, hi in shards)
            # the shards of the unpadded parameters lie inside the padded ones
            for r in range(world):
                lo, hi = shard_bounds(n, world, r)
                assert shards[r][0] <= lo and hi <= shards[r][1] or lo == hi
