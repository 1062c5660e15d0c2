"""Data-parallel packed AdamW with the optimizer state sharded over the ranks
(ZeRO stage 1): every rank holds a replica of the parameters, and the state of
one contiguous shard of them.

The pages' contract is one device ("Packed AdamW / Reference / v1.0.0" code
page, "Execution contract": contiguous FP32 tensors, a dense gradient every
update, one global step).  The update is elementwise, so a rank steps its own
shard exactly as the one-device step would step those elements; what data
parallelism adds around the step is two exchanges of the standard collectives:

  1. reduce-scatter of the flat gradient: rank r receives the sum (or the
     average) over the ranks of elements [r*S, (r+1)*S);
  2. the library's packed step on that shard of the flat parameters, with the
     shard's own state (4 bytes per parameter in the packed modes, so each rank
     keeps 4/world bytes per model parameter);
  3. all-gather of the updated shards into every rank's flat parameters (in
     place: rank r's shard already sits at its place in the output).

The flat buffers hold world*S elements, S a multiple of 4 (every shard keeps
the buffer's 16-byte phase, so the staged kernel copies every shard in bulk);
the padding past the model's parameters is zero and stays zero (a zero
gradient on a zero parameter and zero state gives zero).  `padded_length`
gives the size to allocate; `flatten_into` lays a list of tensors out in such a
buffer.

Nothing here computes any part of the update: the step is the library's
kernel (or `step_fn`, which tests use to put another implementation of the same
step in its place), and the two exchanges are torch.distributed collectives
(NCCL on GPUs).  The reduce-scatter's own arithmetic (the sum over ranks, and
the division of the average) is the collective library's.
"""
from __future__ import annotations

from . import pa_adamw_step_fp32, pa_adamw_step_packed_e4, pa_adamw_step_packed_fp16

ALIGN = 4


def padded_length(n: int, world: int, align: int = ALIGN) -> int:
    """Elements of a flat buffer of n parameters split into world equal shards
    that start on multiples of `align`."""
    if world < 1 or align < 1 or n < 0:
        raise ValueError("bad padded_length request")
    units = -(-max(n, 1) // align)
    return world * (-(-units // world) * align)


def flatten_into(tensors, flat):
    """Copy `tensors` one after the other into the 1-D `flat` (zero past them);
    returns the views of `flat` that hold them, in their shapes."""
    views, off = [], 0
    flat.zero_()
    for t in tensors:
        n = t.numel()
        v = flat[off:off + n]
        v.copy_(t.reshape(-1))
        views.append(v.view(t.shape))
        off += n
    if off > flat.numel():
        raise ValueError("flat buffer too small")
    return views


def _library_step(mode):
    def e4(p, g, state, step, hyper, nonfinite):
        pa_adamw_step_packed_e4(p, g, state[0], step, nonfinite=nonfinite, **hyper)

    def fp16(p, g, state, step, hyper, nonfinite):
        pa_adamw_step_packed_fp16(p, g, state[0], step, nonfinite=nonfinite, **hyper)

    def fp32(p, g, state, step, hyper, nonfinite):
        pa_adamw_step_fp32(p, g, state[0], state[1], step, nonfinite=nonfinite, **hyper)

    return {"e4": e4, "fp16": fp16, "fp32": fp32}[mode]


class ShardedPackedAdamW:
    """ZeRO-1 packed AdamW over a flat parameter buffer of padded_length(n,
    world) FP32 elements (CUDA for the library step).

    step(flat_grads) runs the reduce-scatter, this rank's shard step and the
    all-gather on the current stream; flat_grads has the buffer's length and
    holds this rank's gradient.  average=True averages the gradients over the
    ranks (ReduceOp.AVG), False sums them.  mode: "e4" (default), "fp16" or
    "fp32" as for PackedAdamW.  step_fn(p_shard, g_shard, state, step, hyper,
    nonfinite) replaces the library step (tests).
    """

    def __init__(self, flat_params, group=None, mode: str = "e4", lr: float = 1e-3,
                 betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.01,
                 average: bool = True, step_fn=None):
        import torch
        import torch.distributed as dist

        if mode not in ("e4", "fp16", "fp32"):
            raise ValueError("mode must be 'e4', 'fp16' or 'fp32'")
        if flat_params.dim() != 1 or flat_params.dtype != torch.float32 or \
                not flat_params.is_contiguous():
            raise ValueError("flat_params must be a contiguous 1-D float32 tensor")
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        total = flat_params.numel()
        if total % (self.world * ALIGN) != 0:
            raise ValueError(f"flat_params holds {total} elements: allocate padded_length(n, "
                             f"{self.world}) so that every shard has the same multiple of {ALIGN}")
        self.flat = flat_params
        self.shard = total // self.world
        self.lo = self.rank * self.shard
        self.mode = mode
        self.average = average
        self.hyper = dict(lr=lr, beta1=betas[0], beta2=betas[1], eps=eps, wd=weight_decay)
        self.steps = 0
        dev = flat_params.device
        if mode == "fp32":
            self.state = [torch.zeros(self.shard, dtype=torch.float32, device=dev),
                          torch.zeros(self.shard, dtype=torch.float32, device=dev)]
        else:
            self.state = [torch.zeros(self.shard, dtype=torch.int32, device=dev)]
        self.g_shard = torch.empty(self.shard, dtype=torch.float32, device=dev)
        self.nonfinite = torch.zeros(1, dtype=torch.int64, device=dev)
        self.step_fn = step_fn or _library_step(mode)

    def shard_view(self, flat):
        return flat[self.lo:self.lo + self.shard]

    def step(self, flat_grads):
        import torch.distributed as dist

        if flat_grads.shape != self.flat.shape:
            raise ValueError("flat_grads must match flat_params")
        op = dist.ReduceOp.AVG if self.average else dist.ReduceOp.SUM
        dist.reduce_scatter_tensor(self.g_shard, flat_grads, op=op, group=self.group)
        self.steps += 1
        p = self.shard_view(self.flat)
        self.step_fn(p, self.g_shard, self.state, self.steps, self.hyper, self.nonfinite)
        dist.all_gather_into_tensor(self.flat, p, group=self.group)

    def state_dict(self):
        """This rank's shard of the state, the global step and the layout."""
        return {"steps": self.steps, "world": self.world, "rank": self.rank, "mode": self.mode,
                "state": [s.detach().clone() for s in self.state], "hyper": dict(self.hyper)}

    def load_state_dict(self, sd):
        if (sd["world"], sd["rank"], sd["mode"]) != (self.world, self.rank, self.mode):
            raise ValueError("state of another layout (world, rank or mode)")
        for dst, src in zip(self.state, sd["state"]):
            dst.copy_(src)
        self.steps = int(sd["steps"])
        self.hyper = dict(sd["hyper"])
