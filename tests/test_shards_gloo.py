"""The multi-rank path on the CPU (gloo, world size 2): each rank steps its
own contiguous shard of a flattened parameter space with no collective on the
data path; gathering the shards reproduces the unsharded step bit for bit, and
the timing reduction (max over ranks) works over the process group.  The
per-rank compute here is the CPU oracle (no GPU on this machine); the GPU's
per-shard identity is tested in test_gpu_steps.py
(test_multi_equals_single_and_is_shard_invariant)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import workloads as wl


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, n, mode, out_dir):
    import torch
    import torch.distributed as dist

    import adamw_update_gb300 as pa
    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    align = 2048 if mode == "blockwise" else 4
    lo, hi = pa.shard_bounds(n, world, rank, align)
    p = wl.normal_np(n, 0.02, 1)[lo:hi]
    g = wl.normal_np(n, 1e-3, 2)[lo:hi]
    if mode == "blockwise":
        q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
        m = hi - lo
        nb = -(-m // 2048)
        res = oracle.step_blockwise8(p, g, np.zeros(m, np.uint8), np.zeros(nb, np.float32),
                                     np.zeros(m, np.uint8), np.zeros(nb, np.float32), q1, q2, 3,
                                     **wl.HYPER)
        mine = [res[0].view(np.uint16), res[1], res[2], res[3], res[4]]
    else:
        p1, s1, _ = oracle.step_packed(p, g, np.zeros(hi - lo, np.uint32), 3, **wl.HYPER)
        mine = [p1, s1]
    gathered = [None] * world
    dist.all_gather_object(gathered, (lo, hi, mine))
    t = torch.tensor([float(rank + 1)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        np.save(os.path.join(out_dir, "max.npy"), t.numpy())
        with open(os.path.join(out_dir, "parts.pkl"), "wb") as f:
            import pickle

            pickle.dump(gathered, f)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("mode,n", [("e4", 10_001), ("blockwise", 3 * 2048 + 5)])
def test_two_rank_shards_reassemble_the_unsharded_step(built_package, tmp_path, mode, n):
    import pickle

    import oracle

    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), n, mode, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    assert float(np.load(tmp_path / "max.npy")[0]) == world
    parts = pickle.load(open(tmp_path / "parts.pkl", "rb"))
    assert parts[0][0] == 0 and parts[-1][1] == n
    assert all(parts[k][1] == parts[k + 1][0] for k in range(world - 1))
    p = wl.normal_np(n, 0.02, 1)
    g = wl.normal_np(n, 1e-3, 2)
    if mode == "blockwise":
        q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
        nb = -(-n // 2048)
        whole = oracle.step_blockwise8(p, g, np.zeros(n, np.uint8), np.zeros(nb, np.float32),
                                       np.zeros(n, np.uint8), np.zeros(nb, np.float32), q1, q2,
                                       3, **wl.HYPER)
        whole = [whole[0].view(np.uint16), whole[1], whole[2], whole[3], whole[4]]
        for k in range(5):
            cat = np.concatenate([pt[2][k] for pt in parts])
            assert np.array_equal(cat.view(np.uint8), np.asarray(whole[k]).view(np.uint8)), k
    else:
        p1, s1, _ = oracle.step_packed(p, g, np.zeros(n, np.uint32), 3, **wl.HYPER)
        assert np.array_equal(np.concatenate([pt[2][0] for pt in parts]).view(np.uint32),
                              p1.view(np.uint32))
        assert np.array_equal(np.concatenate([pt[2][1] for pt in parts]), s1)


def test_shard_bounds_cover_and_align(built_package):
    pa = built_package
    for n in (0, 1, 7, 4096, 10_001, 7_000_000_000):
        for world in (1, 2, 3, 8):
            for align in (4, 2048):
                b = [pa.shard_bounds(n, world, r, align) for r in range(world)]
                assert b[0][0] == 0 and b[-1][1] == n
                for (lo, hi), (lo2, _) in zip(b[:-1], b[1:]):
                    assert hi == lo2 and (lo % align == 0 or lo == n)
    with pytest.raises(ValueError):
        pa.shard_bounds(10, 2, 2)
