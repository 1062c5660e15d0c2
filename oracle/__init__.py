"""CPU oracle for the packed-state AdamW update -- test infrastructure only.

The oracle is the plain, slow, scalar C program in ``oracle.c`` (its header
lists the pages and the readings it follows).  This module compiles it with gcc
on first use and wraps it with ctypes and numpy.  Only the tests, the smoke
check and bench.py's CPU-baseline and reference legs may import it: the product
package never does, and the two share no code.

Every wrapper copies its inputs and returns fresh arrays, so callers' arrays
are never modified.  ``threads > 1`` splits the elements (whole 2048-element
blocks in the blockwise mode) into contiguous slices run on Python threads;
ctypes releases the GIL during each call and elements are independent, so the
result is identical to a single-threaded run.

``Oracle(path)`` binds the same wrappers to another build of the C source; the
tests use it to load copies with a planted mistake and check that the pins
catch it.  The module-level functions use the default build.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
TURBO_SOURCE = os.path.join(_HERE, "turbo.c")
_LIB = os.path.join(_HERE, "liboracle.so")
BLOCK = 2048
TURBO_BLOCK = 128
TURBO_MEAN = 64

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_sources(srcs, out: str) -> str:
    """Compile C oracle source files into one shared library at ``out``."""
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, *srcs, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def compile_source(src: str, out: str, turbo: str | None = None) -> str:
    """Compile a copy of oracle.c (``src``) with turbo.c (or ``turbo``, a copy
    of it) into a shared library at ``out``."""
    return compile_sources([src, turbo or TURBO_SOURCE], out)


def build(force: bool = False) -> str:
    """Compile oracle.c and turbo.c into liboracle.so (gcc, strict IEEE binary32)."""
    newest = max(os.path.getmtime(SOURCE), os.path.getmtime(TURBO_SOURCE))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        compile_source(SOURCE, _LIB)
    return _LIB


_f32p = ctypes.POINTER(ctypes.c_float)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64
_d = ctypes.c_double
_HYP = [_i64, _d, _d, _d, _d, _d]  # step, lr, beta1, beta2, eps, wd

_SIGNATURES = {
    "oracle_e4m11_encode_array": (None, [_f32p, _u16p, _i64]),
    "oracle_e4m12_encode_array": (None, [_f32p, _u16p, _i64]),
    "oracle_fp16_encode_array": (None, [_f32p, _u16p, _i64]),
    "oracle_e4m11_decode_array": (None, [_u16p, _f32p, _i64]),
    "oracle_e4m12_decode_array": (None, [_u16p, _f32p, _i64]),
    "oracle_fp16_decode_array": (None, [_u16p, _f32p, _i64]),
    "oracle_bf16_round_array": (None, [_f32p, _u16p, _i64]),
    "oracle_hyperparams": (None, [*_HYP, _f32p]),
    "oracle_adamw_element": (None, [ctypes.c_float] * 4 + [*_HYP, _f32p]),
    "oracle_step_packed_e4": (ctypes.c_uint64, [_f32p, _f32p, _u32p, _i64, *_HYP]),
    "oracle_step_packed_fp16": (ctypes.c_uint64, [_f32p, _f32p, _u32p, _i64, *_HYP]),
    "oracle_step_fp32": (ctypes.c_uint64, [_f32p, _f32p, _f32p, _f32p, _i64, *_HYP]),
    "oracle_encode_state_e4": (ctypes.c_uint64, [_f32p, _f32p, _u32p, _i64]),
    "oracle_decode_state_e4": (None, [_u32p, _f32p, _f32p, _i64]),
    "oracle_encode_state_fp16": (ctypes.c_uint64, [_f32p, _f32p, _u32p, _i64]),
    "oracle_decode_state_fp16": (None, [_u32p, _f32p, _f32p, _i64]),
    "oracle_requantise": (None, [_f32p, _i64, _f32p, _u8p, _f32p]),
    "oracle_step_blockwise8": (
        ctypes.c_uint64,
        [_f32p, _f32p, _u16p, _u8p, _f32p, _u8p, _f32p, _f32p, _f32p, _i64, *_HYP],
    ),
    # TurboAdam-style state (turbo.c)
    "oracle_splitmix64_at": (ctypes.c_uint64, [ctypes.c_uint64, ctypes.c_uint64]),
    "oracle_turbo_uniform_array": (None, [ctypes.c_uint64, _i64, ctypes.c_uint32,
                                          ctypes.POINTER(ctypes.c_uint64), _f32p, _i64]),
    "oracle_q1_levels": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p]),
    "oracle_q1_index_array": (None, [_f32p, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     _f32p, ctypes.POINTER(ctypes.c_int32)]),
    "oracle_q1_endpoints_pair": (None, [_f32p, _i64, ctypes.POINTER(ctypes.c_int32)]),
    "oracle_q1_endpoint_code": (ctypes.c_uint16, [ctypes.c_int]),
    "oracle_q1_endpoint_value": (ctypes.c_int, [ctypes.c_uint16]),
    "oracle_ustate_code_array": (None, [_f32p, _i64, ctypes.c_float, _f32p,
                                        ctypes.POINTER(ctypes.c_int32)]),
    "oracle_turbo_step": (ctypes.c_uint64, [_f32p, _f32p, _i64, _u8p, _u16p, _f32p, _u8p, _u16p,
                                            *_HYP, ctypes.c_uint64]),
    "oracle_turbo_step_at": (ctypes.c_uint64, [_f32p, _f32p, _i64, _u8p, _u16p, _f32p, _u8p, _u16p,
                                               *_HYP, ctypes.c_uint64, ctypes.c_uint64]),
    "oracle_turbo_finalize": (None, [_f32p, _i64, _d]),
    "oracle_turbo_decode": (None, [_i64, _u8p, _u16p, _f32p, _u8p, _u16p, _i64, _d, _d, _d,
                                   _f32p, _f32p]),
}


def _ptr(a: np.ndarray, ctype):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _arr(x, dtype) -> np.ndarray:
    return np.array(x, dtype=dtype, copy=True, order="C").reshape(-1)


def _hyp(step, lr, beta1, beta2, eps, wd):
    return (int(step), float(lr), float(beta1), float(beta2), float(eps), float(wd))


def _slices(n: int, threads: int, align: int = 1):
    """Contiguous [lo, hi) slices, each start a multiple of ``align``."""
    units = -(-n // align)
    threads = max(1, min(int(threads), max(1, units)))
    per = -(-units // threads)
    out = []
    for t in range(threads):
        lo = t * per * align
        hi = min(n, (t + 1) * per * align)
        if lo < hi:
            out.append((lo, hi))
    return out or [(0, n)]


def _run_sliced(fn, n: int, threads: int, align: int = 1) -> int:
    sl = _slices(n, threads, align)
    if len(sl) == 1:
        return int(fn(*sl[0]) or 0)
    results = [0] * len(sl)

    def work(k, lo, hi):
        results[k] = int(fn(lo, hi) or 0)

    ts = [threading.Thread(target=work, args=(k, lo, hi)) for k, (lo, hi) in enumerate(sl)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return sum(results)


class Oracle:
    """ctypes/numpy wrappers over one build of the C oracle."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        lib = ctypes.CDLL(self.path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        self.lib = lib

    # ---- lane codecs ----------------------------------------------------
    def _enc(self, name, x):
        x = _arr(x, np.float32)
        out = np.empty(x.size, np.uint16)
        getattr(self.lib, name)(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), x.size)
        return out

    def _dec(self, name, c):
        c = _arr(c, np.uint16)
        out = np.empty(c.size, np.float32)
        getattr(self.lib, name)(_ptr(c, ctypes.c_uint16), _ptr(out, ctypes.c_float), c.size)
        return out

    def e4m11_encode(self, x):
        """Signed E4M11 codes of FP32 values (first-moment lane)."""
        return self._enc("oracle_e4m11_encode_array", x)

    def e4m12_encode(self, x):
        """Unsigned E4M12 codes of FP32 values (uncorrected-RMS lane)."""
        return self._enc("oracle_e4m12_encode_array", x)

    def fp16_encode(self, x):
        """Saturating binary16 codes of FP32 values (FP16 comparison mode)."""
        return self._enc("oracle_fp16_encode_array", x)

    def e4m11_decode(self, c):
        return self._dec("oracle_e4m11_decode_array", c)

    def e4m12_decode(self, c):
        return self._dec("oracle_e4m12_decode_array", c)

    def fp16_decode(self, c):
        return self._dec("oracle_fp16_decode_array", c)

    def bf16_round(self, x):
        """bfloat16 bit patterns of FP32 values, round to nearest even."""
        return self._enc("oracle_bf16_round_array", x)

    def hyperparams(self, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01):
        """The eight FP32 scalars (b1, b2, c1, c2, bc2, ss, dk, ef)."""
        out = np.empty(8, np.float32)
        self.lib.oracle_hyperparams(*_hyp(step, lr, beta1, beta2, eps, wd),
                                    _ptr(out, ctypes.c_float))
        return out

    def adamw_element(self, p, g, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                      wd=0.01):
        """(p', m', v') of one FP32 element."""
        out = np.empty(3, np.float32)
        self.lib.oracle_adamw_element(
            ctypes.c_float(p), ctypes.c_float(g), ctypes.c_float(m), ctypes.c_float(v),
            *_hyp(step, lr, beta1, beta2, eps, wd), _ptr(out, ctypes.c_float))
        return out

    # ---- state-word codecs ----------------------------------------------
    def encode_state(self, m, rms, mode="e4"):
        """Pack (m, rms) into uint32 words; returns (words, nonfinite_count)."""
        m = _arr(m, np.float32)
        rms = _arr(rms, np.float32)
        assert m.size == rms.size
        w = np.empty(m.size, np.uint32)
        fn = getattr(self.lib, f"oracle_encode_state_{mode}")
        bad = fn(_ptr(m, ctypes.c_float), _ptr(rms, ctypes.c_float),
                 _ptr(w, ctypes.c_uint32), m.size)
        return w, int(bad)

    def decode_state(self, words, mode="e4"):
        """Unpack uint32 words into (m, rms) FP32 arrays."""
        w = _arr(words, np.uint32)
        m = np.empty(w.size, np.float32)
        r = np.empty(w.size, np.float32)
        fn = getattr(self.lib, f"oracle_decode_state_{mode}")
        fn(_ptr(w, ctypes.c_uint32), _ptr(m, ctypes.c_float), _ptr(r, ctypes.c_float), w.size)
        return m, r

    # ---- steps ----------------------------------------------------------
    def step_packed(self, p, g, state, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                    wd=0.01, mode="e4", threads=1):
        """One packed step (mode 'e4' or 'fp16'); returns (p', state', nonfinite)."""
        p = _arr(p, np.float32)
        g = _arr(g, np.float32)
        s = _arr(state, np.uint32)
        assert p.size == g.size == s.size
        fn = self.lib.oracle_step_packed_e4 if mode == "e4" else self.lib.oracle_step_packed_fp16
        hy = _hyp(step, lr, beta1, beta2, eps, wd)

        def run(lo, hi):
            return fn(_ptr(p[lo:hi], ctypes.c_float), _ptr(g[lo:hi], ctypes.c_float),
                      _ptr(s[lo:hi], ctypes.c_uint32), hi - lo, *hy)

        bad = _run_sliced(run, p.size, threads)
        return p, s, bad

    def step_fp32(self, p, g, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01,
                  threads=1):
        """One FP32-moment step; returns (p', m', v', nonfinite)."""
        p, g, m, v = (_arr(a, np.float32) for a in (p, g, m, v))
        assert p.size == g.size == m.size == v.size
        hy = _hyp(step, lr, beta1, beta2, eps, wd)
        fn = self.lib.oracle_step_fp32

        def run(lo, hi):
            return fn(*(_ptr(a[lo:hi], ctypes.c_float) for a in (p, g, m, v)), hi - lo, *hy)

        bad = _run_sliced(run, p.size, threads)
        return p, m, v, bad

    def requantise(self, x, qmap):
        """Blockwise nearest-entry codes and per-block absmax of FP32 values."""
        x = _arr(x, np.float32)
        q = _arr(qmap, np.float32)
        assert q.size == 256
        nb = -(-x.size // BLOCK)
        code = np.empty(x.size, np.uint8)
        amax = np.empty(nb, np.float32)
        self.lib.oracle_requantise(_ptr(x, ctypes.c_float), x.size, _ptr(q, ctypes.c_float),
                                   _ptr(code, ctypes.c_uint8), _ptr(amax, ctypes.c_float))
        return code, amax

    def step_blockwise8(self, p, g, m_code, m_absmax, v_code, v_absmax, qmap1, qmap2, step,
                        lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01, threads=1):
        """One 8-bit blockwise step.

        Returns (p_bf16_bits uint16, m_code', m_absmax', v_code', v_absmax', nonfinite).
        """
        p = _arr(p, np.float32)
        g = _arr(g, np.float32)
        mc = _arr(m_code, np.uint8)
        vc = _arr(v_code, np.uint8)
        ma = _arr(m_absmax, np.float32)
        va = _arr(v_absmax, np.float32)
        q1 = _arr(qmap1, np.float32)
        q2 = _arr(qmap2, np.float32)
        n = p.size
        nb = -(-n // BLOCK)
        assert g.size == n and mc.size == n and vc.size == n and ma.size == nb and va.size == nb
        assert q1.size == 256 and q2.size == 256
        out = np.empty(n, np.uint16)
        hy = _hyp(step, lr, beta1, beta2, eps, wd)
        fn = self.lib.oracle_step_blockwise8

        def run(lo, hi):
            b0 = lo // BLOCK
            return fn(_ptr(p[lo:hi], ctypes.c_float), _ptr(g[lo:hi], ctypes.c_float),
                      _ptr(out[lo:hi], ctypes.c_uint16), _ptr(mc[lo:hi], ctypes.c_uint8),
                      _ptr(ma[b0:], ctypes.c_float), _ptr(vc[lo:hi], ctypes.c_uint8),
                      _ptr(va[b0:], ctypes.c_float), _ptr(q1, ctypes.c_float),
                      _ptr(q2, ctypes.c_float), hi - lo, *hy)

        bad = _run_sliced(run, n, threads, align=BLOCK)
        return out, mc, ma, vc, va, bad


def turbo_state_sizes(n: int):
    """Element counts of the TurboAdam-style state arrays of an n-element tensor:
    ucode (uint8), umean (uint16 bf16), uscal (float32), vidx (uint8), vend
    (uint16 fp16)."""
    return {"ucode": -(-n // 4), "umean": -(-n // TURBO_MEAN), "uscal": 3,
            "vidx": -(-n // 2), "vend": 2 * -(-n // TURBO_BLOCK)}


def turbo_zero_state(n: int):
    """The initial state (everything zero): decodes to m = v = 0."""
    z = turbo_state_sizes(n)
    return {"ucode": np.zeros(z["ucode"], np.uint8), "umean": np.zeros(z["umean"], np.uint16),
            "uscal": np.zeros(3, np.float32), "vidx": np.zeros(z["vidx"], np.uint8),
            "vend": np.zeros(z["vend"], np.uint16)}


def _turbo_methods():
    def splitmix64_at(self, seed, counter):
        return int(self.lib.oracle_splitmix64_at(ctypes.c_uint64(seed), ctypes.c_uint64(counter)))

    def turbo_uniform(self, seed, step, stream, index):
        idx = _arr(index, np.uint64)
        out = np.empty(idx.size, np.float32)
        self.lib.oracle_turbo_uniform_array(ctypes.c_uint64(seed), int(step), int(stream),
                                            _ptr(idx, ctypes.c_uint64), _ptr(out, ctypes.c_float),
                                            idx.size)
        return out

    def q1_levels(self, lo, hi, bits=4):
        out = np.empty(1 << bits, np.float32)
        self.lib.oracle_q1_levels(int(lo), int(hi), int(bits), _ptr(out, ctypes.c_float))
        return out

    def q1_index(self, v, lo, hi, u, bits=4):
        v = _arr(v, np.float32)
        u = _arr(u, np.float32)
        out = np.empty(v.size, np.int32)
        self.lib.oracle_q1_index_array(_ptr(v, ctypes.c_float), v.size, int(lo), int(hi),
                                       int(bits), _ptr(u, ctypes.c_float),
                                       _ptr(out, ctypes.c_int32))
        return out

    def q1_endpoints(self, v):
        v = _arr(v, np.float32)
        out = np.empty(2, np.int32)
        self.lib.oracle_q1_endpoints_pair(_ptr(v, ctypes.c_float), v.size,
                                          _ptr(out, ctypes.c_int32))
        return int(out[0]), int(out[1])

    def q1_endpoint_code(self, e):
        return int(self.lib.oracle_q1_endpoint_code(int(e)))

    def q1_endpoint_value(self, h):
        return int(self.lib.oracle_q1_endpoint_value(int(h)))

    def ustate_code(self, r, s, u):
        r = _arr(r, np.float32)
        u = _arr(u, np.float32)
        out = np.empty(r.size, np.int32)
        self.lib.oracle_ustate_code_array(_ptr(r, ctypes.c_float), r.size, ctypes.c_float(s),
                                          _ptr(u, ctypes.c_float), _ptr(out, ctypes.c_int32))
        return out

    def turbo_step(self, p, g, state, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                   wd=0.01, seed=0x12345678, index0=0):
        """One TurboAdam-style step of one tensor; returns (p', state', nonfinite)
        with state a dict of ucode, umean, uscal, vidx, vend (copied).  index0:
        the arrays are the slice of a larger tensor from element index0 (a
        multiple of 128) on, whose rounding counters take the tensor's indices."""
        assert index0 % TURBO_BLOCK == 0
        p = _arr(p, np.float32)
        g = _arr(g, np.float32)
        n = p.size
        assert g.size == n
        st = {k: _arr(v, v.dtype) for k, v in state.items()}
        z = turbo_state_sizes(n)
        for k, size in z.items():
            assert st[k].size == size, (k, st[k].size, size)
        bad = self.lib.oracle_turbo_step_at(
            _ptr(p, ctypes.c_float), _ptr(g, ctypes.c_float), n, _ptr(st["ucode"], ctypes.c_uint8),
            _ptr(st["umean"], ctypes.c_uint16), _ptr(st["uscal"], ctypes.c_float),
            _ptr(st["vidx"], ctypes.c_uint8), _ptr(st["vend"], ctypes.c_uint16),
            *_hyp(step, lr, beta1, beta2, eps, wd), ctypes.c_uint64(seed), ctypes.c_uint64(index0))
        return p, st, int(bad)

    def turbo_decode(self, state, n, step, beta1=0.9, beta2=0.999, eps=1e-8):
        """(m_prev, v_dec): the prior moments the step at `step` decodes."""
        st = {k: _arr(v, v.dtype) for k, v in state.items()}
        m = np.empty(n, np.float32)
        v = np.empty(n, np.float32)
        self.lib.oracle_turbo_decode(
            int(n), _ptr(st["ucode"], ctypes.c_uint8), _ptr(st["umean"], ctypes.c_uint16),
            _ptr(st["uscal"], ctypes.c_float), _ptr(st["vidx"], ctypes.c_uint8),
            _ptr(st["vend"], ctypes.c_uint16), int(step), float(beta1), float(beta2), float(eps),
            _ptr(m, ctypes.c_float), _ptr(v, ctypes.c_float))
        return m, v

    def turbo_finalize(self, uscal, n, factor=1.1):
        s = _arr(uscal, np.float32)
        self.lib.oracle_turbo_finalize(_ptr(s, ctypes.c_float), int(n), float(factor))
        return s

    for f in (splitmix64_at, turbo_uniform, q1_levels, q1_index, q1_endpoints, q1_endpoint_code,
              q1_endpoint_value, ustate_code, turbo_step, turbo_decode, turbo_finalize):
        setattr(Oracle, f.__name__, f)


_turbo_methods()

_default: Oracle | None = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
    return _default


def __getattr__(name):
    # module-level access to the default build's wrappers: oracle.step_packed(...)
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(default(), name)
