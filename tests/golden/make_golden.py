"""Writes the stored expected values under tests/golden/ by calling the CPU
oracle only (never the CUDA path).  Run from the repository root:

    python tests/golden/make_golden.py

single4096_trajectory.json: the single-tensor workload (4,096 parameters,
p ~ N(0, 0.02) seed 0, g ~ N(0, 1e-3) drawn fresh each step with seed 1000+t,
zero state, lr 1e-3, betas (0.9, 0.999), eps 1e-8, wd 0.01), 10 steps in the
packed E4, packed FP16 and FP32 modes.  For each step it stores the SHA-256 of
the parameter and state bytes and the first eight values, so a later change to
the oracle's arithmetic shows up as a changed fixture.
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as wl  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def sha(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def trajectory():
    n, hy = 4096, wl.HYPER
    p0 = wl.normal_np(n, 0.02, 0)
    out = {}
    for mode in ("e4", "fp16", "fp32"):
        p = p0.copy()
        st = [np.zeros(n, np.uint32)] if mode != "fp32" else [np.zeros(n, np.float32)] * 2
        steps = []
        for t in range(1, 11):
            g = wl.normal_np(n, 1e-3, 1000 + t)
            if mode == "fp32":
                p, m, v, bad = oracle.step_fp32(p, g, st[0], st[1], t, **hy)
                st = [m, v]
            else:
                p, s, bad = oracle.step_packed(p, g, st[0], t, mode=mode, **hy)
                st = [s]
            steps.append({
                "step": t,
                "nonfinite": bad,
                "sha256": sha(p, *st),
                "p_head_bits": [int(x) for x in p[:8].view(np.uint32)],
                "state_head_bits": [int(x) for x in np.asarray(st[0][:8]).view(np.uint32)],
            })
        out[mode] = steps
    return out


if __name__ == "__main__":
    doc = {
        "source": "written by tests/golden/make_golden.py from the CPU oracle only",
        "workload": "single-4096: p~N(0,0.02) seed 0; g~N(0,1e-3) seed 1000+t; zero state; "
                    "lr 1e-3, betas (0.9, 0.999), eps 1e-8, wd 0.01; 10 steps",
        "modes": trajectory(),
    }
    with open(os.path.join(HERE, "single4096_trajectory.json"), "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote single4096_trajectory.json")
