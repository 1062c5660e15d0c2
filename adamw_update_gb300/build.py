"""Build libpackedadam.so (and its contracted-arithmetic variant) for sm_103a.

    python adamw_update_gb300/build.py

libpackedadam.so       the product library: every binary32 operation of the
                       update rounds once (no FMA contraction, IEEE division
                       and square root, subnormals kept), so its results are
                       bit-identical to a strict binary32 evaluation.
libpackedadam_fast.so  the same source with PA_FAST_MATH: the decoupled-decay
                       line p*(1-lr*wd) - upd is one FMA (a tolerance build:
                       parameters within 2 ulp of the largest term, state
                       words unchanged).

Both are compiled in parallel with one -gencode (sm_103a) and linked against
the static CUDA runtime; host code is built with -ffp-contract=off so the
double-precision hyperparameter scalars round the same on x86 and Arm.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "packedadam.cu")
DEPS = [SRC, os.path.join(ROOT, "include", "packedadam.h")] + [
    os.path.join(HERE, "csrc", f) for f in ("codecs.cuh", "blockwise.cuh", "pipeline.cuh",
                                              "f32x2.cuh", "turbo.cuh", "exact.cuh")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-I", os.path.join(ROOT, "include"),
          "-Xcompiler", "-fPIC,-ffp-contract=off", "-shared"]
VARIANTS = {
    "libpackedadam.so": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false"],
    "libpackedadam_fast.so": ["-DPA_FAST_MATH", "-fmad=true", "-ftz=false"],
}


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpackedadam")
    return path


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, extra: list[str] | None = None, verbose: bool = False) -> dict:
    """Compile both variants (in parallel); returns {name: path}."""
    procs = {}
    outs = {}
    for name, flags in VARIANTS.items():
        out = os.path.join(HERE, name)
        outs[name] = out
        if not (force or extra or _stale(out)):
            continue
        tmp = out + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, *COMMON, *flags, *(extra or []), SRC, "-o", tmp]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs[name] = (subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), tmp, out)
    failed = []
    for name, (proc, tmp, out) in procs.items():
        log = proc.communicate()[0].decode(errors="replace")
        if proc.returncode != 0:
            failed.append(f"{name}:\n{log}")
        else:
            os.replace(tmp, out)
            if verbose and log.strip():
                print(log)
    if failed:
        raise RuntimeError("nvcc failed\n" + "\n".join(failed))
    return outs


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
