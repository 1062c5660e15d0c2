"""PackedAdamW: a torch.optim.Optimizer over libpackedadam.so's tensor-list steps.

"Packed AdamW Reference" README v1.0.0 lists a reusable dense optimizer
interface and, for its trainer, a latest-only exact-resume checkpoint and a
smoke check of a one-word state ledger; the code page's "Execution contract"
fixes contiguous CUDA FP32 parameters on one device, a dense gradient for every
parameter on every update, one parameter group and one global step.  This
class keeps that contract:

* ``mode="e4"`` (default): one int32 tensor of packed words per parameter
  (E4M11 first moment low, E4M12 uncorrected RMS high), 4 bytes per parameter;
  ``"fp16"``: the FP16-first/FP16-RMS words; ``"fp32"``: ordinary FP32 m and v.
* ``step()`` runs ONE kernel launch over every parameter of the group.
* the non-finite count of every update accumulates on the device
  (``nonfinite_count()`` reads it).
* ``state_dict()`` holds the state tensors and the global step;
  ``load_state_dict()`` restores them bit for bit, so training continues exactly
  as if uninterrupted (``save_checkpoint`` / ``load_checkpoint`` write and read
  a latest-only checkpoint file atomically).

Cost of moving gradients.  The step hands the library the list of (p, g,
state) pointers; the library keeps one device descriptor table per distinct
list (64 at most, least recently used freed first).  A list it has not seen
costs a cudaMalloc and a synchronous upload, and past 64 lists each new one
also a cudaFree, which waits for the device.  Gradients that move between
steps -- ``zero_grad(set_to_none=True)``, torch's default, lets backward
allocate new ones, which the caching allocator often but not always puts at
the same addresses -- can therefore make a step synchronise the host.  Keep
gradients in place (``zero_grad(set_to_none=False)``, or gradient buckets)
to pay the upload once; in mode "e4" with up to 1024 parameters on one
stream, ``pa_adamw_step_packed_e4_multi_noalloc`` is a step that never
allocates or waits, whatever the pointers.
"""
from __future__ import annotations

import os

import torch

from . import (pa_adamw_step_fp32_multi, pa_adamw_step_packed_e4_multi,
               pa_adamw_step_packed_fp16_multi, tensor_list)

_STEP = {"e4": pa_adamw_step_packed_e4_multi, "fp16": pa_adamw_step_packed_fp16_multi,
         "fp32": pa_adamw_step_fp32_multi}


class PackedAdamW(torch.optim.Optimizer):
    def __init__(self, params, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-8,
                 weight_decay: float = 0.01, mode: str = "e4"):
        if mode not in _STEP:
            raise ValueError(f"mode must be one of {sorted(_STEP)}")
        if not 0.0 <= betas[0] < 1.0 or not 0.0 <= betas[1] < 1.0 or eps < 0.0:
            raise ValueError("betas must lie in [0, 1) and eps must be >= 0")
        defaults = dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                        mode=mode, step=0)
        super().__init__(params, defaults)
        if len(self.param_groups) != 1:
            raise ValueError("PackedAdamW takes one parameter group (one global step)")
        device = None
        for p in self.param_groups[0]["params"]:
            if not (p.is_cuda and p.dtype == torch.float32 and p.is_contiguous()):
                raise ValueError("parameters must be contiguous CUDA float32 tensors")
            if device is not None and p.device != device:
                raise ValueError("parameters must live on one device")
            device = p.device
        self._nonfinite = torch.zeros(1, dtype=torch.int64, device=device)
        self._cache_key = None
        self._cache_arr = None

    # ---- state ----------------------------------------------------------------
    def _state_of(self, p):
        st = self.state[p]
        if not st:
            mode = self.param_groups[0]["mode"]
            if mode == "fp32":
                st["exp_avg"] = torch.zeros_like(p)
                st["exp_avg_sq"] = torch.zeros_like(p)
            else:
                st["packed"] = torch.zeros(p.shape, dtype=torch.int32, device=p.device)
        return st

    def load_state_dict(self, state_dict):
        """torch's loader casts every state tensor of a floating-point parameter
        to the parameter's dtype, which would turn the packed int32 words into
        float32 numbers; the words are set aside and restored unchanged."""
        import copy

        sd = copy.copy(state_dict)
        sd["state"] = {k: dict(v) for k, v in state_dict["state"].items()}
        words = {k: v.pop("packed") for k, v in sd["state"].items() if "packed" in v}
        super().load_state_dict(sd)
        ids = [pid for g in state_dict["param_groups"] for pid in g["params"]]
        params = [p for g in self.param_groups for p in g["params"]]
        for pid, p in zip(ids, params):
            if pid in words:
                self.state[p]["packed"] = words[pid].to(device=p.device, dtype=torch.int32,
                                                        copy=True)
        self._cache_key = None

    def state_bytes(self) -> int:
        """Bytes of persistent optimizer state (4 per parameter in the packed modes)."""
        return sum(t.numel() * t.element_size() for st in self.state.values()
                   for t in st.values() if torch.is_tensor(t))

    def nonfinite_count(self) -> int:
        """Elements with a non-finite new p, m or v, summed over all updates."""
        return int(self._nonfinite.item())

    # ---- the update -----------------------------------------------------------
    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        group = self.param_groups[0]
        mode = group["mode"]
        entries = []
        for p in group["params"]:
            if p.grad is None:
                raise RuntimeError("PackedAdamW needs a dense gradient for every parameter")
            if p.grad.is_sparse or not p.grad.is_contiguous() or p.grad.dtype != torch.float32:
                raise RuntimeError("gradients must be dense contiguous float32")
            st = self._state_of(p)
            if mode == "fp32":
                entries.append((p, p.grad, st["exp_avg"], st["exp_avg_sq"]))
            else:
                entries.append((p, p.grad, st["packed"]))
        key = tuple(t.data_ptr() for e in entries for t in e)
        if key != self._cache_key:  # the ctypes list is rebuilt only when a pointer moves
            self._cache_arr = tensor_list(entries, fp32=mode == "fp32")
            self._cache_key = key
        group["step"] += 1
        beta1, beta2 = group["betas"]
        _STEP[mode](self._cache_arr, group["step"], lr=group["lr"], beta1=beta1, beta2=beta2,
                    eps=group["eps"], wd=group["weight_decay"], nonfinite=self._nonfinite)
        return loss


_PLAIN = (type(None), bool, int, float, str, bytes, torch.Tensor)


def _check_plain(x, where="extra"):
    """Checkpoints are read back with torch.load(weights_only=True), which
    unpickles tensors and plain containers only; refuse anything else when
    saving rather than writing a file that cannot be loaded."""
    if isinstance(x, _PLAIN):
        return
    if isinstance(x, (list, tuple)):
        for k, v in enumerate(x):
            _check_plain(v, f"{where}[{k}]")
        return
    if isinstance(x, dict):
        for k, v in x.items():
            _check_plain(k, f"{where} key")
            _check_plain(v, f"{where}[{k!r}]")
        return
    raise TypeError(f"{where}: {type(x).__name__} is not plain data (None, bool, int, float, "
                    "str, bytes, tensors, and lists, tuples and dicts of them)")


def save_checkpoint(path: str, params, optimizer: PackedAdamW, extra=None) -> None:
    """Write a latest-only checkpoint (parameters, optimizer state, global
    step) atomically: a temporary file renamed over `path`.  `extra` must be
    plain data (see _check_plain): the loader unpickles nothing else."""
    _check_plain(extra)
    blob = {"params": [p.detach().clone() for p in params],
            "optimizer": optimizer.state_dict(), "extra": extra}
    tmp = f"{path}.tmp.{os.getpid()}"
    torch.save(blob, tmp)
    os.replace(tmp, path)


def load_checkpoint(path: str, params, optimizer: PackedAdamW):
    """Restore parameters and optimizer state written by save_checkpoint, bit
    for bit; returns the `extra` object that was saved.  The file is read with
    torch.load(weights_only=True): tensors and plain containers only, so a file
    holding any other pickled object is refused before anything is restored."""
    blob = torch.load(path, map_location="cpu", weights_only=True)
    with torch.no_grad():
        for p, saved in zip(params, blob["params"]):
            p.copy_(saved)
    optimizer.load_state_dict(blob["optimizer"])
    return blob["extra"]
