"""adamw_update_gb300 -- AdamW with packed, quantized persistent moment state on
NVIDIA GB300 (sm_103a).

A thin ctypes binding over libpackedadam.so (C ABI in include/packedadam.h).
Each function has the name of its C entry point and only marshals arguments:
torch CUDA tensors become device pointers, the stream defaults to torch's
current stream, and a non-zero status raises PackedAdamError with the
library's message.  Every step of the update runs in the library's kernels;
there is no fallback.  Importing the package loads the library and fails with
ImportError if it has not been built (python adamw_update_gb300/build.py).

Sources: "Packed AdamW Reference" README v1.0.0, "The canonical format"
(one uint32 word per FP32 parameter: E4M11 first moment low, E4M12
uncorrected RMS high); "Packed AdamW / Reference / v1.0.0", "Release scope"
and "Execution contract"; KBench "quantized-optimizer-state" reference.py,
quantized_adamw_step (8-bit blockwise mode).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "PackedAdamError", "library_path", "pa_version", "pa_status_string",
    "pa_encode_state", "pa_decode_state", "pa_encode_state_fp16", "pa_decode_state_fp16",
    "pa_adamw_step_packed_e4", "pa_adamw_step_packed_fp16", "pa_adamw_step_fp32",
    "pa_adamw_step_blockwise8", "pa_adamw_step_packed_e4_multi",
    "pa_adamw_step_packed_fp16_multi", "pa_adamw_step_fp32_multi", "pa_release_tables",
    "shard_bounds", "pa_adamw_step_packed_e4_multi_noalloc", "pa_adamw_step_packed_e4_host",
    "pa_hyper_table_fill", "pa_adamw_step_packed_e4_multi_graph",
    "pa_adamw_step_packed_e4_bf16g", "pa_adamw_step_packed_e4_multi_bf16g", "pa_shutdown",
    "pa_adamw_step_blockwise8_multi", "pa_device_fault", "pa_turbo_step", "turbo_state",
]

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path(fast: bool = False) -> str:
    return os.path.join(_HERE, "libpackedadam_fast.so" if fast else "libpackedadam.so")


class PackedAdamError(RuntimeError):
    def __init__(self, status: int, name: str, message: str):
        super().__init__(f"{name}: {message}")
        self.status = status


class PaTensor(ctypes.Structure):
    """pa_tensor: {float* p; const float* g; void* state; void* state2; int64 n}."""
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("state", ctypes.c_void_p),
                ("state2", ctypes.c_void_p), ("n", ctypes.c_int64)]


_vp, _i64, _i32, _d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
_HYP = [_i64, _d, _d, _d, _d, _d]  # step, lr, beta1, beta2, eps, wd
_SIGNATURES = {
    "pa_version": (_i32, []),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_encode_state": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "pa_decode_state": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "pa_encode_state_fp16": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "pa_decode_state_fp16": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "pa_adamw_step_packed_e4": (_i32, [_vp, _vp, _vp, _i64, *_HYP, _vp, _vp]),
    "pa_adamw_step_packed_fp16": (_i32, [_vp, _vp, _vp, _i64, *_HYP, _vp, _vp]),
    "pa_adamw_step_fp32": (_i32, [_vp, _vp, _vp, _vp, _i64, *_HYP, _vp, _vp]),
    "pa_adamw_step_blockwise8": (_i32, [_vp] * 9 + [_i64, *_HYP, _vp, _vp]),
    "pa_adamw_step_packed_e4_multi": (_i32, [ctypes.POINTER(PaTensor), _i32, *_HYP, _vp, _vp]),
    "pa_adamw_step_packed_fp16_multi": (_i32, [ctypes.POINTER(PaTensor), _i32, *_HYP, _vp, _vp]),
    "pa_adamw_step_fp32_multi": (_i32, [ctypes.POINTER(PaTensor), _i32, *_HYP, _vp, _vp]),
    "pa_release_tables": (_i32, []),
}


def load_library(path: str) -> ctypes.CDLL:
    """Load a build of libpackedadam.so and declare its C signatures."""
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


# PA_LIBRARY_VARIANT=fast selects the contracted-arithmetic build of the same source
_PATH = library_path(fast=os.environ.get("PA_LIBRARY_VARIANT", "") == "fast")
if not os.path.exists(_PATH):
    raise ImportError(f"{_PATH} is missing: build it with "
                      "`python adamw_update_gb300/build.py` (needs nvcc)")
_lib = load_library(_PATH)


def _check(status: int):
    if status != 0:
        name = _lib.pa_status_string(status).decode()
        raise PackedAdamError(status, name, _lib.pa_last_error().decode())


def _ptr(t, dtype=None):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (device memory)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected dtype {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _hyp(step, lr, beta1, beta2, eps, wd):
    return (int(step), float(lr), float(beta1), float(beta2), float(eps), float(wd))


def _t():
    import torch

    return torch


def pa_version() -> int:
    return _lib.pa_version()


def pa_status_string(status: int) -> str:
    return _lib.pa_status_string(status).decode()


# ---- codecs -----------------------------------------------------------------

def pa_encode_state(m, rms, word, nonfinite=None, stream=None):
    """word[i] = E4M12(rms[i]) << 16 | E4M11(m[i])."""
    torch = _t()
    _check(_lib.pa_encode_state(_ptr(m, torch.float32), _ptr(rms, torch.float32),
                                _ptr(word, torch.int32), m.numel(), _ptr(nonfinite),
                                _stream(stream)))


def pa_decode_state(word, m, rms, stream=None):
    torch = _t()
    _check(_lib.pa_decode_state(_ptr(word, torch.int32), _ptr(m, torch.float32),
                                _ptr(rms, torch.float32), word.numel(), _stream(stream)))


def pa_encode_state_fp16(m, rms, word, nonfinite=None, stream=None):
    torch = _t()
    _check(_lib.pa_encode_state_fp16(_ptr(m, torch.float32), _ptr(rms, torch.float32),
                                     _ptr(word, torch.int32), m.numel(), _ptr(nonfinite),
                                     _stream(stream)))


def pa_decode_state_fp16(word, m, rms, stream=None):
    torch = _t()
    _check(_lib.pa_decode_state_fp16(_ptr(word, torch.int32), _ptr(m, torch.float32),
                                     _ptr(rms, torch.float32), word.numel(), _stream(stream)))


# ---- single-tensor steps (state words are int32 tensors holding uint32 bits) --

def pa_adamw_step_packed_e4(p, g, state, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                            wd=0.0, nonfinite=None, stream=None):
    torch = _t()
    _check(_lib.pa_adamw_step_packed_e4(_ptr(p, torch.float32), _ptr(g, torch.float32),
                                        _ptr(state, torch.int32), p.numel(),
                                        *_hyp(step, lr, beta1, beta2, eps, wd),
                                        _ptr(nonfinite), _stream(stream)))


def pa_adamw_step_packed_fp16(p, g, state, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                              wd=0.0, nonfinite=None, stream=None):
    torch = _t()
    _check(_lib.pa_adamw_step_packed_fp16(_ptr(p, torch.float32), _ptr(g, torch.float32),
                                          _ptr(state, torch.int32), p.numel(),
                                          *_hyp(step, lr, beta1, beta2, eps, wd),
                                          _ptr(nonfinite), _stream(stream)))


def pa_adamw_step_fp32(p, g, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0,
                       nonfinite=None, stream=None):
    torch = _t()
    _check(_lib.pa_adamw_step_fp32(_ptr(p, torch.float32), _ptr(g, torch.float32),
                                   _ptr(m, torch.float32), _ptr(v, torch.float32), p.numel(),
                                   *_hyp(step, lr, beta1, beta2, eps, wd),
                                   _ptr(nonfinite), _stream(stream)))


def pa_adamw_step_blockwise8(p, g, p_bf16, m_code, m_absmax, v_code, v_absmax, qmap1, qmap2,
                             step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01,
                             nonfinite=None, stream=None):
    torch = _t()
    _check(_lib.pa_adamw_step_blockwise8(
        _ptr(p, torch.float32), _ptr(g, torch.float32), _ptr(p_bf16, torch.bfloat16),
        _ptr(m_code, torch.uint8), _ptr(m_absmax, torch.float32), _ptr(v_code, torch.uint8),
        _ptr(v_absmax, torch.float32), _ptr(qmap1, torch.float32), _ptr(qmap2, torch.float32),
        p.numel(), *_hyp(step, lr, beta1, beta2, eps, wd), _ptr(nonfinite), _stream(stream)))


# ---- multi-tensor steps --------------------------------------------------------

def tensor_list(entries, fp32: bool = False, grad_dtype=None):
    """ctypes pa_tensor array from (p, g, state) or (p, g, m, v) tuples;
    grad_dtype: torch.float32 (default) or torch.bfloat16 for the *_bf16g calls."""
    torch = _t()
    gd = torch.float32 if grad_dtype is None else grad_dtype
    arr = (PaTensor * len(entries))()
    for k, e in enumerate(entries):
        if fp32:
            p, g, m, v = e
            arr[k] = PaTensor(_ptr(p, torch.float32), _ptr(g, gd),
                              _ptr(m, torch.float32), _ptr(v, torch.float32), p.numel())
        else:
            p, g, s = e
            arr[k] = PaTensor(_ptr(p, torch.float32), _ptr(g, gd),
                              _ptr(s, torch.int32), None, p.numel())
    return arr


def _multi(fn, entries, fp32, step, lr, beta1, beta2, eps, wd, nonfinite, stream):
    arr = entries if isinstance(entries, ctypes.Array) else tensor_list(entries, fp32)
    _check(fn(arr, len(arr), *_hyp(step, lr, beta1, beta2, eps, wd), _ptr(nonfinite),
              _stream(stream)))


def pa_adamw_step_packed_e4_multi(entries, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                  wd=0.0, nonfinite=None, stream=None):
    """One launch over a list of (p, g, state) tensors (or a tensor_list array)."""
    _multi(_lib.pa_adamw_step_packed_e4_multi, entries, False, step, lr, beta1, beta2, eps, wd,
           nonfinite, stream)


def pa_adamw_step_packed_fp16_multi(entries, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                    wd=0.0, nonfinite=None, stream=None):
    _multi(_lib.pa_adamw_step_packed_fp16_multi, entries, False, step, lr, beta1, beta2, eps,
           wd, nonfinite, stream)


def pa_adamw_step_fp32_multi(entries, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0,
                             nonfinite=None, stream=None):
    """One launch over a list of (p, g, m, v) tensors (or a tensor_list array)."""
    _multi(_lib.pa_adamw_step_fp32_multi, entries, True, step, lr, beta1, beta2, eps, wd,
           nonfinite, stream)


def pa_release_tables():
    _check(_lib.pa_release_tables())


_lib.pa_shutdown.restype = _i32
_lib.pa_shutdown.argtypes = []


def pa_shutdown():
    _check(_lib.pa_shutdown())


# ---- sharding of a flattened parameter space ------------------------------------

def shard_bounds(n: int, world: int, rank: int, align: int = 4):
    """[lo, hi) of rank's contiguous shard of n elements split over world ranks.

    Shards start on multiples of `align` (4 elements keeps every shard's
    16-byte phase equal to the whole buffer's; use 2048 for the blockwise mode
    so no quantisation block is split).  Elements are independent, so stepping
    each shard on its own rank gives the same bits as stepping the whole; the
    step itself needs no collective (gradients arrive by reduce-scatter and
    parameters leave by all-gather, outside this library).
    """
    if world < 1 or not 0 <= rank < world or align < 1 or n < 0:
        raise ValueError("bad shard request")
    units = -(-n // align)
    per = -(-units // world) * align
    lo = min(n, rank * per)
    return lo, min(n, lo + per)


# ---- the multi-tensor packed-E4 step that allocates nothing -------------------

_lib.pa_adamw_step_packed_e4_multi_noalloc.restype = _i32
_lib.pa_adamw_step_packed_e4_multi_noalloc.argtypes = [
    ctypes.POINTER(PaTensor), _i32, *_HYP, _vp, _vp]


def pa_adamw_step_packed_e4_multi_noalloc(entries, step, lr=1e-3, beta1=0.9, beta2=0.999,
                                          eps=1e-8, wd=0.0, nonfinite=None, stream=None):
    """pa_adamw_step_packed_e4_multi without any device allocation by the
    library, for callers whose device memory is owned by their own allocator
    or who must not meet cudaMalloc's synchronisation: the descriptor table
    goes to a fixed device array of 1024 entries.  Calls that overlap on the
    GPU race on that array; the first call on a device should come before any
    stream capture."""
    _multi(_lib.pa_adamw_step_packed_e4_multi_noalloc, entries, False, step, lr, beta1, beta2,
           eps, wd, nonfinite, stream)


# ---- the packed-E4 step over host-resident tensors ------------------------------

_lib.pa_adamw_step_packed_e4_host.restype = _i32
_lib.pa_adamw_step_packed_e4_host.argtypes = [_vp, _vp, _vp, _i64, *_HYP, _vp, _i64, _vp, _vp]


def _host_ptr(t, dtype):
    if t.is_cuda:
        raise ValueError("expected a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if t.dtype != dtype:
        raise TypeError(f"expected dtype {dtype}, got {t.dtype}")
    return t.data_ptr()


def pa_adamw_step_packed_e4_host(p, g, state, workspace, step, lr=1e-3, beta1=0.9, beta2=0.999,
                                 eps=1e-8, wd=0.0, nonfinite=None, stream=None):
    """Packed-E4 step over host tensors.  Pinned tensors are read and written
    in place by the step kernel over the host link; otherwise they are
    streamed through the CUDA tensor `workspace` (uint8, >= 2.36 MB; larger
    means longer chunks), which is checked either way.  Synchronise `stream`
    before reading p or state."""
    torch = _t()
    _check(_lib.pa_adamw_step_packed_e4_host(
        _host_ptr(p, torch.float32), _host_ptr(g, torch.float32), _host_ptr(state, torch.int32),
        p.numel(), *_hyp(step, lr, beta1, beta2, eps, wd), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(nonfinite), _stream(stream)))


# ---- graph-replayable step: device table of per-step scalars ----------------------

HYPER_ROW_FLOATS = 8  # pa_hyper: b1, b2, c1, c2, bc2, ss, dk, ef

_lib.pa_hyper_table_fill.restype = _i32
_lib.pa_hyper_table_fill.argtypes = [_vp, _i64, _i32, _vp, _d, _d, _d, _d, _d, _vp]
_lib.pa_adamw_step_packed_e4_multi_graph.restype = _i32
_lib.pa_adamw_step_packed_e4_multi_graph.argtypes = [
    ctypes.POINTER(PaTensor), _i32, _vp, _i32, _vp, _vp, _vp, _vp]


def pa_hyper_table_fill(rows, first_step, count, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                        wd=0.0, lr_per_step=None, stream=None):
    """Fill `rows` (CUDA float32 tensor of >= count*8 floats) with the scalars of
    steps first_step .. first_step+count-1; lr_per_step: optional schedule."""
    torch = _t()
    if rows.numel() < count * HYPER_ROW_FLOATS:
        raise ValueError("rows holds fewer than count rows")
    sched = None
    if lr_per_step is not None:
        sched = (ctypes.c_double * count)(*[float(x) for x in lr_per_step])
    _check(_lib.pa_hyper_table_fill(_ptr(rows, torch.float32), int(first_step), int(count), sched,
                                    float(lr), float(beta1), float(beta2), float(eps), float(wd),
                                    _stream(stream)))


def pa_adamw_step_packed_e4_multi_graph(entries, rows, nrows, index, status=None, nonfinite=None,
                                        stream=None):
    """Packed-E4 list step with the scalars of row index[0] of `rows`, then
    index[0] += 1 on the device (capturable in a CUDA graph)."""
    torch = _t()
    arr = entries if isinstance(entries, ctypes.Array) else tensor_list(entries)
    _check(_lib.pa_adamw_step_packed_e4_multi_graph(
        arr, len(arr), _ptr(rows, torch.float32), int(nrows), _ptr(index, torch.int64),
        _ptr(status, torch.int32) if status is not None else None, _ptr(nonfinite),
        _stream(stream)))


# ---- packed-E4 steps with bfloat16 gradients --------------------------------------

_lib.pa_adamw_step_packed_e4_bf16g.restype = _i32
_lib.pa_adamw_step_packed_e4_bf16g.argtypes = [_vp, _vp, _vp, _i64, *_HYP, _vp, _vp]
_lib.pa_adamw_step_packed_e4_multi_bf16g.restype = _i32
_lib.pa_adamw_step_packed_e4_multi_bf16g.argtypes = [ctypes.POINTER(PaTensor), _i32, *_HYP, _vp, _vp]


def pa_adamw_step_packed_e4_bf16g(p, g, state, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                  wd=0.0, nonfinite=None, stream=None):
    """Packed-E4 step with a torch.bfloat16 gradient (widened exactly)."""
    torch = _t()
    _check(_lib.pa_adamw_step_packed_e4_bf16g(_ptr(p, torch.float32), _ptr(g, torch.bfloat16),
                                              _ptr(state, torch.int32), p.numel(),
                                              *_hyp(step, lr, beta1, beta2, eps, wd),
                                              _ptr(nonfinite), _stream(stream)))


def pa_adamw_step_packed_e4_multi_bf16g(entries, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                        wd=0.0, nonfinite=None, stream=None):
    """One launch over (p, g_bf16, state) tuples (or a tensor_list array made
    with grad_dtype=torch.bfloat16)."""
    torch = _t()
    arr = entries if isinstance(entries, ctypes.Array) else \
        tensor_list(entries, grad_dtype=torch.bfloat16)
    _check(_lib.pa_adamw_step_packed_e4_multi_bf16g(arr, len(arr),
                                                    *_hyp(step, lr, beta1, beta2, eps, wd),
                                                    _ptr(nonfinite), _stream(stream)))


# ---- blockwise tensor-list step ----------------------------------------------------

class PaBlockwiseTensor(ctypes.Structure):
    """pa_blockwise_tensor: p, g, p_bf16, m_code, m_absmax, v_code, v_absmax, n."""
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("p_bf16", ctypes.c_void_p),
                ("m_code", ctypes.c_void_p), ("m_absmax", ctypes.c_void_p),
                ("v_code", ctypes.c_void_p), ("v_absmax", ctypes.c_void_p), ("n", ctypes.c_int64)]


_lib.pa_adamw_step_blockwise8_multi.restype = _i32
_lib.pa_adamw_step_blockwise8_multi.argtypes = [ctypes.POINTER(PaBlockwiseTensor), _i32, _vp, _vp,
                                                *_HYP, _vp, _vp]


def blockwise_list(entries):
    """ctypes pa_blockwise_tensor array from (p, g, p_bf16, m_code, m_absmax,
    v_code, v_absmax) tuples of CUDA tensors."""
    torch = _t()
    arr = (PaBlockwiseTensor * len(entries))()
    for k, (p, g, pb, mc, ma, vc, va) in enumerate(entries):
        arr[k] = PaBlockwiseTensor(_ptr(p, torch.float32), _ptr(g, torch.float32),
                                   _ptr(pb, torch.bfloat16), _ptr(mc, torch.uint8),
                                   _ptr(ma, torch.float32), _ptr(vc, torch.uint8),
                                   _ptr(va, torch.float32), p.numel())
    return arr


def pa_adamw_step_blockwise8_multi(entries, qmap1, qmap2, step, lr=1e-3, beta1=0.9, beta2=0.999,
                                   eps=1e-8, wd=0.01, nonfinite=None, stream=None):
    """One launch of the blockwise step over a list of tensors."""
    torch = _t()
    arr = entries if isinstance(entries, ctypes.Array) else blockwise_list(entries)
    _check(_lib.pa_adamw_step_blockwise8_multi(arr, len(arr), _ptr(qmap1, torch.float32),
                                               _ptr(qmap2, torch.float32),
                                               *_hyp(step, lr, beta1, beta2, eps, wd),
                                               _ptr(nonfinite), _stream(stream)))


# ---- fault flag of the staged step kernels ------------------------------------------

_lib.pa_device_fault.restype = _i32
_lib.pa_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint32), _i32]


def pa_device_fault(clear: bool = False) -> int:
    """0 if no bounded wait of a staged step kernel has run out on the current
    device since the flag was last cleared, else its fault code (1-3)."""
    code = ctypes.c_uint32(0)
    _check(_lib.pa_device_fault(ctypes.byref(code), 1 if clear else 0))
    return int(code.value)


# ---- TurboAdam-style step (UState first moment, 1Q second moment) -----------------

class PaTurboState(ctypes.Structure):
    """pa_turbo_state: device pointers of ucode, umean, uscal, vidx, vend."""
    _fields_ = [("ucode", ctypes.c_void_p), ("umean", ctypes.c_void_p), ("uscal", ctypes.c_void_p),
                ("vidx", ctypes.c_void_p), ("vend", ctypes.c_void_p)]


_lib.pa_turbo_step.restype = _i32
_lib.pa_turbo_step.argtypes = [_vp, _vp, _i64, ctypes.POINTER(PaTurboState), *_HYP, _d,
                               ctypes.c_uint64, _vp, _vp]

TURBO_BLOCK = 128
TURBO_MEAN = 64


def turbo_state(n: int, device="cuda"):
    """Zero TurboAdam-style state of an n-element tensor (the initial state):
    dict of ucode uint8, umean int16 (bf16 bits), uscal float32[3], vidx uint8,
    vend int16 (fp16 bits)."""
    torch = _t()
    return {"ucode": torch.zeros(-(-n // 4), dtype=torch.uint8, device=device),
            "umean": torch.zeros(-(-n // TURBO_MEAN), dtype=torch.int16, device=device),
            "uscal": torch.zeros(3, dtype=torch.float32, device=device),
            "vidx": torch.zeros(-(-n // 2), dtype=torch.uint8, device=device),
            "vend": torch.zeros(2 * -(-n // TURBO_BLOCK), dtype=torch.int16, device=device)}


def pa_turbo_step(p, g, state, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0,
                  m_step_factor=1.1, seed=0x12345678, nonfinite=None, stream=None):
    """TurboAdam-style step of one tensor: p updated in place, `state` (from
    turbo_state) advanced, scales rotated."""
    torch = _t()
    st = PaTurboState(_ptr(state["ucode"], torch.uint8), _ptr(state["umean"], torch.int16),
                      _ptr(state["uscal"], torch.float32), _ptr(state["vidx"], torch.uint8),
                      _ptr(state["vend"], torch.int16))
    _check(_lib.pa_turbo_step(_ptr(p, torch.float32), _ptr(g, torch.float32), p.numel(),
                              ctypes.byref(st), *_hyp(step, lr, beta1, beta2, eps, wd),
                              float(m_step_factor), ctypes.c_uint64(seed), _ptr(nonfinite),
                              _stream(stream)))
