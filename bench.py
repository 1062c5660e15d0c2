"""Benchmark of the packed-E4 AdamW step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--mode e4|fp16|fp32] [--impl ours|reference] [--no-e2e]

One step is one pass of the whole hot path over one batch of synthetic input:
the multi-tensor packed step (one persistent launch over the workload's
tensor list) with inputs resident in HBM.  The default workload is flat-7e9:
one FP32 tensor of 7e9 parameters (28 GB each for p, g and the state words;
g = 1e-3 * t(df=3) with a 1e-4 fraction scaled by 1e4), 3 warm-up and 20
timed steps.  Every step moves 140 GB, far more than the 129 MB L2, so no
flush is needed; workloads whose bytes per step are under 4x the L2 get an
L2 flush (a 512 MB write) between timed steps, outside the timed launch.

Printed (rank 0, one JSON line): params/s of the whole job (the units every
rank processed / the slowest rank's time), the roofline of the step kernel
against the measured HBM copy bandwidth, the CPU oracle on a bounded sample
of the same workload (cpu_baseline), the end-to-end rate through the public
API with host buffers (host-to-device copies of p, g and the state, the step,
device-to-host copies of p and the state, all inside the timed region), and
the SM clocks sampled during the timed region.

N > 1 (torchrun): each rank steps its own shard of the same size on its own
GPU (elements are independent, so no collective is on the data path); a
barrier and a max-reduction of the timings are the only communication.

The default line (flat-7e9, packed E4, N = 1) also carries `configs`: every
workload of the benchmark measured the same way after the headline, each with
its own buffers, warm-up, timed steps and oracle baseline -- single-4096 (10
steps), gpt-52 packed E4 and FP32 (100 steps each), gpt2-148 packed E4 and FP16
(50 steps each), flat-7e9 (the headline's numbers), the 8-bit blockwise
mode on 1e9 parameters (20 steps) and the TurboAdam-style step on GPT-2
small's 124M parameters (20 steps).

--impl reference times the CPU oracle, as it stands, on this machine's cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

# TurboAdam-style: read p, g, 2-bit codes, 4-bit indices, a bf16 mean per 64 and two
# fp16 endpoints per 128; write all but g
TURBO_BYTES = 4 + 4 + 0.25 + 0.5 + 2 / 64 + 4 / 128 + 4 + 0.25 + 0.5 + 2 / 64 + 4 / 128
BYTES_PER_PARAM = {"e4": 20, "fp16": 20, "fp32": 28, "blockwise": 14 + 16 / 2048,
                   "turbo": TURBO_BYTES}
KERNEL_NAME = {"e4": "adamw_step_pipe_kernel<0>", "fp16": "adamw_step_pipe_kernel<1>",
               "fp32": "adamw_step_pipe_kernel<2>", "blockwise": "blockwise8_pipe_kernel<false>",
               "turbo": "turbo_step_kernel"}
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="flat-7e9", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--mode", default="e4", choices=["e4", "fp16", "fp32"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--fast", action="store_true", help="use libpackedadam_fast.so")
    ap.add_argument("--grad", default="fp32", choices=["fp32", "bf16"],
                    help="gradient dtype of the packed-E4 step (bf16: 18 bytes per parameter)")
    ap.add_argument("--graph", action="store_true",
                    help="packed E4: capture the step (device-indexed scalar rows) in a CUDA "
                         "graph and time its replays")
    ap.add_argument("--op", default="step", choices=["step", "encode", "decode"],
                    help="encode/decode: time the standalone E4 state codecs (12 B/param) on "
                         "the one-tensor workload instead of the step")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration measurements (the `configs` object)")
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0,
                    help="oracle seconds per configuration's cpu_baseline")
    ap.add_argument("--params", type=int, default=None,
                    help="override the parameter count of a one-tensor workload (flat-7e9, "
                         "blockwise-1e9): the same distributions at another size, for profiling")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_code_digest_input() -> str:
    """The kernel sources with // comments and blank lines removed: the traffic
    record stays valid across comment edits, not across code changes."""
    import re

    src = os.path.join(ROOT, "adamw_update_gb300", "csrc")
    out = []
    for name in ("packedadam.cu", "codecs.cuh", "blockwise.cuh", "pipeline.cuh", "f32x2.cuh",
                 "turbo.cuh", "exact.cuh"):
        with open(os.path.join(src, name)) as f:
            for line in f:
                code = re.sub(r"//.*$", "", line).rstrip()
                if code:
                    out.append(code)
    return "\n".join(out)


def traffic_per_param(mode):
    """DRAM bytes per parameter of the step kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256(kernel_code_digest_input().encode())
    entry = d.get(mode)
    if not entry or entry.get("source_sha256") != h.hexdigest():
        return None
    return float(entry["dram_bytes_per_param"])


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    QUERY = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            bus = f[1].lower()
            if self.bus_id and not (bus.endswith(self.bus_id[-12:]) or self.bus_id.endswith(bus[-12:])):
                continue
            try:
                mhz.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(mhz), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Workload construction (device buffers, seeded; outside every timed region)
# ---------------------------------------------------------------------------

PARAMS_OVERRIDE = {}


def tensor_sizes(name):
    if name == "gpt-52":
        return [n for _, n in wl.GPT52_SHAPES]
    if name == "gpt2-148":
        return [n for _, n in wl.GPT2_148_SHAPES]
    return [PARAMS_OVERRIDE.get(name, wl.WORKLOADS[name]["n"])]


def fill_gradient_(name, g, sizes, seed):
    if name == "flat-7e9":
        wl.fill_student_t_saturating_(g, seed)
    elif name == "gpt2-148":
        wl.fill_gpt2_grads_(g, sizes, seed)
    else:
        wl.fill_normal_(g, 1e-3, seed, stream=1)


class Workload:
    """Flat device buffers for a workload; tensors are contiguous slices."""

    def __init__(self, name, mode, device, seed):
        import torch

        self.name, self.mode = name, mode
        self.grad_bf16 = False
        self.sizes = tensor_sizes(name)
        self.n = sum(self.sizes)
        n = self.n
        f32 = torch.float32
        if name == "turbo-124m":
            import adamw_update_gb300 as pa

            self.mode = "turbo"
            self.p = wl.fill_normal_(torch.empty(n, dtype=f32, device=device), 0.02, seed)
            self.g = wl.fill_turbo_grads_(torch.empty(n, dtype=f32, device=device), seed)
            self.st = pa.turbo_state(n, device)
            self.fresh_g = None
            return
        if name == "blockwise-1e9":
            self.mode = mode = "blockwise"
            q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
            nb = wl.blocks(n)
            self.p = wl.fill_normal_(torch.empty(n, dtype=f32, device=device), 0.02, seed)
            self.g = torch.empty(n, dtype=f32, device=device)
            wl.fill_normal_(self.g, 1e-3, seed, stream=1)
            self.p_bf16 = torch.empty(n, dtype=torch.bfloat16, device=device)
            self.m_code = torch.full((n,), wl.nearest_zero_code(q1), dtype=torch.uint8, device=device)
            self.v_code = torch.full((n,), wl.nearest_zero_code(q2), dtype=torch.uint8, device=device)
            self.m_absmax = torch.zeros(nb, dtype=f32, device=device)
            self.v_absmax = torch.zeros(nb, dtype=f32, device=device)
            self.q1 = torch.from_numpy(q1).to(device)
            self.q2 = torch.from_numpy(q2).to(device)
            return
        self.p = wl.fill_normal_(torch.empty(n, dtype=f32, device=device), 0.02, seed)
        self.g = torch.empty(n, dtype=f32, device=device)
        fill_gradient_(name, self.g, self.sizes, seed)
        if mode == "fp32":
            self.s = [torch.zeros(n, dtype=f32, device=device), torch.zeros(n, dtype=f32, device=device)]
        else:
            self.s = [torch.zeros(n, dtype=torch.int32, device=device)]
        self.fresh_g = None
        if name == "single-4096":  # the workload draws g afresh every step
            self.fresh_g = []

    def bytes_per_param(self):
        return BYTES_PER_PARAM[self.mode] - (2 if self.grad_bf16 else 0)

    def bytes_per_step(self):
        return self.bytes_per_param() * self.n

    def tensor_array(self, pa, g=None):
        g = self.g if g is None else g
        offs = np.cumsum([0] + self.sizes)
        ents = []
        for a, b in zip(offs[:-1], offs[1:]):
            ents.append((self.p[a:b], g[a:b], *[s[a:b] for s in self.s]))
        import torch

        return pa.tensor_list(ents, fp32=self.mode == "fp32",
                              grad_dtype=torch.bfloat16 if self.grad_bf16 else None)


def step_fn(pa, w, hy, nonfinite):
    """A closure running one step on torch's current stream."""
    import torch

    if w.mode == "blockwise":
        def run(t):
            pa.pa_adamw_step_blockwise8(w.p, w.g, w.p_bf16, w.m_code, w.m_absmax, w.v_code,
                                        w.v_absmax, w.q1, w.q2, t, nonfinite=nonfinite, **hy)
        return run
    if w.mode == "turbo":
        def run(t):
            pa.pa_turbo_step(w.p, w.g, w.st, t, nonfinite=nonfinite, **hy)
        return run
    fn = {"e4": pa.pa_adamw_step_packed_e4_multi, "fp16": pa.pa_adamw_step_packed_fp16_multi,
          "fp32": pa.pa_adamw_step_fp32_multi}[w.mode]
    if w.grad_bf16:
        fn = pa.pa_adamw_step_packed_e4_multi_bf16g
    arrays = [w.tensor_array(pa)]
    if w.fresh_g is not None:
        arrays = []
        for k in range(64):
            gk = torch.empty_like(w.g)
            wl.fill_normal_(gk, 1e-3, seed=1000 + k, stream=1)
            w.fresh_g.append(gk)
            arrays.append(w.tensor_array(pa, gk))

    def run(t):
        fn(arrays[t % len(arrays)], t, nonfinite=nonfinite, **hy)
    return run


def graph_step_fn(pa, w, hy, nonfinite, nsteps):
    """One step = one replay of a CUDA graph holding the device-indexed packed
    E4 list step; the scalar rows of steps 1..nsteps are filled beforehand."""
    import torch

    if w.mode != "e4" or w.fresh_g is not None or w.grad_bf16:
        raise SystemExit("--graph applies to the packed-E4 workloads with a fixed FP32 gradient")
    rows = torch.empty(nsteps * pa.HYPER_ROW_FLOATS, dtype=torch.float32, device=w.p.device)
    pa.pa_hyper_table_fill(rows, 1, nsteps, **hy)
    index = torch.zeros(1, dtype=torch.int64, device=w.p.device)
    status = torch.zeros(1, dtype=torch.int32, device=w.p.device)
    arr = w.tensor_array(pa)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # makes the descriptor table before capture
        pa.pa_adamw_step_packed_e4_multi_graph(arr, rows, nsteps, index, status, nonfinite)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.pa_adamw_step_packed_e4_multi_graph(arr, rows, nsteps, index, status, nonfinite)
    index.zero_()  # replays start again at step 1

    def run(t):
        graph.replay()
    return run


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------

def oracle_sample_rate(arrays, mode, seconds, threads, q=None):
    """Time the oracle (as it stands, `threads` host threads) on a bounded
    sample; repeats whole passes until `seconds` have elapsed (at least one).
    Returns (params/s, elements per pass, passes)."""
    import oracle

    hy = wl.HYPER
    n = arrays[0].size
    passes, t0 = 0, time.perf_counter()
    st = [a.copy() if isinstance(a, np.ndarray) else {k: v.copy() for k, v in a.items()}
          for a in arrays]
    while True:
        passes += 1
        if mode == "turbo":  # one thread: the oracle's step is sequential
            p, g, ts = st
            p, ts, _ = oracle.turbo_step(p, g, ts, passes, **hy)
            ts["uscal"] = oracle.turbo_finalize(ts["uscal"], p.size)
            st = [p, g, ts]
        elif mode == "blockwise":
            p, g, mc, ma, vc, va = st
            ob, mc, ma, vc, va, _ = oracle.step_blockwise8(p, g, mc, ma, vc, va, q[0], q[1],
                                                           passes, threads=threads, **hy)
            st = [p, g, mc, ma, vc, va]
        elif mode == "fp32":
            st[0], st[2], st[3], _ = oracle.step_fp32(st[0], st[1], st[2], st[3], passes,
                                                      threads=threads, **hy)
        else:
            st[0], st[2], _ = oracle.step_packed(st[0], st[1], st[2], passes, mode=mode,
                                                 threads=threads, **hy)
        el = time.perf_counter() - t0
        if el >= seconds:
            return n * passes / el, n, passes


def sample_size(mode, seconds, threads, total):
    """Elements for about `seconds` of oracle work on `threads` threads,
    calibrated on a 2^20-element run, capped at 2^27 and at the workload."""
    import oracle

    k = 1 << 20
    rng = np.random.default_rng(0)
    p = rng.normal(0, 0.02, k).astype(np.float32)
    g = rng.normal(0, 1e-3, k).astype(np.float32)
    if mode == "turbo":
        k = 1 << 16
        p, g = p[:k], g[:k]
    t0 = time.perf_counter()
    if mode == "turbo":
        oracle.turbo_step(p, g, oracle.turbo_zero_state(k), 1)
    elif mode == "fp32":
        z = np.zeros(k, np.float32)
        oracle.step_fp32(p, g, z, z, 1, threads=threads)
    elif mode == "blockwise":
        z8 = np.zeros(k, np.uint8)
        za = np.zeros(k // 2048, np.float32)
        q = wl.dynamic_qmap_signed()
        oracle.step_blockwise8(p, g, z8, za, z8, za, q, q, 1, threads=threads)
    else:
        oracle.step_packed(p, g, np.zeros(k, np.uint32), 1, mode=mode, threads=threads)
    rate = k / max(time.perf_counter() - t0, 1e-6)
    s = int(min(total, 1 << 27, max(1 << 16 if mode == "turbo" else 1 << 20, rate * seconds)))
    return (s // 2048) * 2048 if s >= 2048 else s


def sample_gradient(name, s, seed):
    """Host FP32 gradient sample of s elements with the workload's distribution."""
    import torch

    g = torch.empty(s, dtype=torch.float32)
    if name == "gpt2-148":
        sizes, left = [], s
        for n in tensor_sizes(name):
            if left == 0:
                break
            sizes.append(min(n, left))
            left -= sizes[-1]
        return wl.fill_gpt2_grads_(g, sizes, seed)
    fill_gradient_(name, g, [s], seed)
    return g


def host_sample(w, s):
    """First s elements of the workload's inputs, as host numpy arrays."""
    if w.mode == "turbo":
        import oracle

        return [w.p[:s].cpu().numpy(), w.g[:s].cpu().numpy(), oracle.turbo_zero_state(s)], None
    if w.mode == "blockwise":
        nb = wl.blocks(s)
        arrays = [w.p[:s].cpu().numpy(), w.g[:s].cpu().numpy(), w.m_code[:s].cpu().numpy(),
                  w.m_absmax[:nb].cpu().numpy(), w.v_code[:s].cpu().numpy(),
                  w.v_absmax[:nb].cpu().numpy()]
        return arrays, (w.q1.cpu().numpy(), w.q2.cpu().numpy())
    arrays = [w.p[:s].cpu().numpy(), w.g[:s].float().cpu().numpy()]  # bf16 widens exactly
    for st in w.s:
        a = st[:s].cpu().numpy()
        arrays.append(a.view(np.uint32) if a.dtype == np.int32 else a)
    return arrays, None


def host_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        return None
    return None


def prefix_sample(arrays, mode, s):
    """The first s elements of a host sample (s whole 2048-blocks, or all of it,
    in the blockwise mode, whose absmax arrays are per block)."""
    if mode == "blockwise":
        nb = wl.blocks(s)
        p, g, mc, ma, vc, va = arrays
        return [p[:s], g[:s], mc[:s], ma[:nb], vc[:s], va[:nb]]
    if mode == "turbo":
        import oracle

        return [arrays[0][:s], arrays[1][:s], oracle.turbo_zero_state(s)]
    return [a[:s] for a in arrays]


def cpu_baseline(w, seconds):
    """The oracle on all host cores for `seconds`, then on one thread for a
    quarter of that on a prefix of the same sample."""
    cores = host_cores() if w.mode != "turbo" else 1
    s = sample_size(w.mode, seconds / 4, cores, w.n)
    arrays, q = host_sample(w, s)
    rate, n, passes = oracle_sample_rate(arrays, w.mode, seconds, cores, q)
    s1 = min(s, max(2048, int(rate / cores * seconds / 8) // 2048 * 2048))
    rate1, n1, passes1 = oracle_sample_rate(prefix_sample(arrays, w.mode, s1), w.mode,
                                            seconds / 4, 1, q)
    return {"value": rate, "unit": "params/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} parameters of the {w.name} workload, {passes} oracle "
                      f"steps in {cores} host threads",
            "single_thread": {"value": rate1, "unit": "params/s",
                              "sample": f"first {n1} parameters, {passes1} oracle steps "
                                        f"in 1 thread"}}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def time_launches(run, first_step, steps, flush, stream):
    """CUDA events on the launching stream around each of `steps` launches
    (steps first_step, first_step+1, ...), an L2 flush between launches when
    `flush` is a buffer (outside the launch's events), and events around the
    whole region.  Returns (per-launch ms, region ms)."""
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    first = torch.cuda.Event(enable_timing=True)
    last = torch.cuda.Event(enable_timing=True)
    first.record(stream)
    for k in range(steps):
        if flush is not None:
            flush.fill_(float(k))
        starts[k].record(stream)
        run(first_step + k)
        ends[k].record(stream)
    last.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], first.elapsed_time(last)


def l2_policy(w, flush):
    return ("flushed between steps (512 MB write)" if flush is not None
            else f"inputs larger than L2 ({w.bytes_per_step() / 1e9:.1f} GB per step)")


def kernel_name(w, graph=False):
    if w.grad_bf16:
        return "adamw_step_pipe_kernel<0,bfloat16>"
    return "adamw_step_table_kernel<0>" if graph else KERNEL_NAME[w.mode]


def run_codec(lib, args, device):
    """pa_encode_state or pa_decode_state over the one-tensor workload: m and
    the RMS from the oracle-free seeded generators (m ~ N(0, 1e-3), RMS =
    |N(0, 1e-3)|), words from encoding them; 12 bytes per parameter (read 8,
    write 4 to encode; read 4, write 8 to decode)."""
    import torch

    if args.workload not in ("flat-7e9", "blockwise-1e9"):
        raise SystemExit("--op encode/decode applies to the one-tensor workloads")
    n = tensor_sizes(args.workload)[0]
    m = wl.fill_normal_(torch.empty(n, dtype=torch.float32, device=device), 1e-3, 5)
    r = wl.fill_normal_(torch.empty(n, dtype=torch.float32, device=device), 1e-3, 6).abs_()
    w = torch.empty(n, dtype=torch.int32, device=device)
    lib.pa_encode_state(m, r, w)
    if args.op == "encode":
        def run(t):
            lib.pa_encode_state(m, r, w)
    else:
        def run(t):
            lib.pa_decode_state(w, m, r)
    stream = torch.cuda.current_stream()
    for t in range(args.warmup):
        run(t)
    torch.cuda.synchronize()
    launch_ms, _ = time_launches(run, 0, args.steps, None, stream)
    kernel_ms = statistics.mean(launch_ms)
    peak, peak_kind = measured_peak()
    achieved = 12 * n / (kernel_ms / 1e3) / 1e9
    name = "encode_state_kernel<0>" if args.op == "encode" else "decode_state_kernel<0>"
    line = {"metric": f"E4 state {args.op}: params/s and HBM GB/s", "value": n / (kernel_ms / 1e3),
            "unit": "params/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kernel_ms, "higher_is_better": True, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload if args.params is None
                       else f"{args.workload} at {n} params", "op": args.op,
                       "bytes_per_param": 12,
                       "l2": f"inputs larger than L2 ({12 * n / 1e9:.1f} GB per step)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind, "kernel": name,
                         "kernel_ms": kernel_ms,
                         "kernel_ms_median": statistics.median(launch_ms)},
            "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.fast:
        os.environ["PA_LIBRARY_VARIANT"] = "fast"
    import adamw_update_gb300 as lib

    if args.op != "step":
        if world > 1:
            raise SystemExit("--op encode/decode runs on one GPU")
        run_codec(lib, args, device)
        return
    line = headline(lib, args, device, world, rank)
    if rank == 0 and world == 1 and want_configs(args):
        import gc

        gc.collect()
        torch.cuda.empty_cache()
        line["configs"] = measure_configs(lib, args, device, line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def headline(lib, args, device, world, rank):
    """The bench line's workload: timed steps, roofline, e2e, cpu_baseline,
    clocks.  Returns the line (rank 0) or None; every device buffer it made is
    released when it returns."""
    import torch
    import torch.distributed as dist

    w = Workload(args.workload, args.mode, device, seed=1234 + rank)
    hy = wl.HYPER
    nonfinite = torch.zeros(1, dtype=torch.int64, device=device)
    if args.grad == "bf16":
        if w.mode != "e4":
            raise SystemExit("--grad bf16 applies to the packed-E4 mode")
        w.g = w.g.to(torch.bfloat16)
        w.grad_bf16 = True
    run = step_fn(lib, w, hy, nonfinite)
    if args.graph:
        run = graph_step_fn(lib, w, hy, nonfinite, args.warmup + args.steps + 2)
    stream = torch.cuda.current_stream()
    flush = None
    if w.bytes_per_step() < 4 * L2_BYTES:
        flush = torch.empty(512 * 2 ** 20 // 4, dtype=torch.float32, device=device)

    for t in range(1, args.warmup + 1):
        run(t)
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(device)
    sampler = ClockSampler(getattr(props, "pci_bus_id", None) and
                           f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0")
    sampler.start()
    time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launch_ms, region_ms = time_launches(run, args.warmup + 1, args.steps, flush, stream)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = statistics.mean(launch_ms) if flush is not None else region_ms / args.steps
    kernel_ms = statistics.mean(launch_ms)
    median_ms = statistics.median(launch_ms)
    t = torch.tensor([step_ms, kernel_ms, median_ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    step_ms, kernel_ms, median_ms = float(t[0]), float(t[1]), float(t[2])

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(lib, w, hy, args, stream, nonfinite)
        if world > 1:
            et = torch.tensor([e2e["_ms"]], dtype=torch.float64, device=device)
            dist.all_reduce(et, op=dist.ReduceOp.MAX)
            e2e["_ms"] = float(et[0])
        e2e_ms = e2e.pop("_ms")
        e2e["value"] = None if e2e_ms != e2e_ms else w.n * world / (e2e_ms / 1e3)

    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(w, args.cpu_seconds)
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    bpp = w.bytes_per_param()
    achieved = bpp * w.n / (kernel_ms / 1e3) / 1e9
    traffic = None if w.grad_bf16 else traffic_per_param(w.mode)
    return {
        "metric": "packed-E4 AdamW step: params/s and HBM GB/s as % of GB300 peak, 1 GPU"
                  if w.mode == "e4" else f"{w.mode} AdamW step: params/s and HBM GB/s",
        "value": w.n * world / (step_ms / 1e3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": w.name if args.params is None else f"{w.name} at {w.n} params",
            "mode": w.mode, "params_per_gpu": w.n,
            "tensors": len(w.sizes), "bytes_per_param": bpp,
            "l2": l2_policy(w, flush),
            "parallelism": f"{world} independent shards, no data-path collective",
            "library": "libpackedadam_fast.so" if args.fast else "libpackedadam.so",
            "grad": args.grad,
            "launch": "CUDA graph replay" if args.graph else "C-ABI call per step",
        },
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": peak_kind,
            "traffic": None if traffic is None else traffic * w.n,
            "kernel": kernel_name(w, args.graph),
            "kernel_ms": kernel_ms,
            "kernel_ms_median": median_ms,
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (2 if args.graph else 1),
        "clocks": clocks,
        "nonfinite": int(nonfinite.item()),
    }


# The five workloads of the benchmark, each measured on its own after the
# headline (flat-7e9 is the headline itself): (workload, mode, timed steps).
CONFIGS = [
    ("single-4096", "e4", 10),
    ("gpt-52", "e4", 100),
    ("gpt-52", "fp32", 100),
    ("gpt2-148", "e4", 50),
    ("gpt2-148", "fp16", 50),
    ("flat-7e9", "e4", None),
    ("blockwise-1e9", "blockwise", 20),
    ("turbo-124m", "turbo", 20),
]


def want_configs(args):
    return not (args.no_configs or args.params is not None or args.graph or args.fast
                or args.grad != "fp32" or args.workload != "flat-7e9" or args.mode != "e4"
                or args.op != "step")


def measure_configs(lib, args, device, head):
    """Every workload of CONFIGS, one after the other, each with its own device
    buffers (released before the next), 3 warm-up steps, CUDA events around
    each timed launch, an L2 flush between launches when its bytes per step
    are under 4x the L2, and the oracle on a bounded sample of it."""
    out = {}
    for name, mode, steps in CONFIGS:
        key = f"{name}/{mode}"
        if steps is None:  # the headline's own numbers
            r = head["roofline"]
            out[key] = {"workload": name, "mode": mode, "params": head["config"]["params_per_gpu"],
                        "tensors": head["config"]["tensors"], "steps": head["steps"],
                        "warmup": head["warmup"], "us_per_step": head["ms_per_step"] * 1e3,
                        "params_per_s": head["value"], "gb_s": r["achieved"], "frac": r["frac"],
                        "kernel": r["kernel"], "kernel_ms": r["kernel_ms"],
                        "kernel_ms_median": r["kernel_ms_median"], "l2": head["config"]["l2"],
                        "cpu_baseline": head["cpu_baseline"], "measured": "the headline"}
            continue
        out[key] = measure_config(lib, name, mode, steps, max(3, args.warmup), device,
                                  args.config_cpu_seconds)
    return out


def measure_config(lib, name, mode, steps, warmup, device, cpu_seconds):
    import torch

    w = Workload(name, mode, device, seed=1234)
    nonfinite = torch.zeros(1, dtype=torch.int64, device=device)
    run = step_fn(lib, w, wl.HYPER, nonfinite)
    stream = torch.cuda.current_stream()
    flush = None
    if w.bytes_per_step() < 4 * L2_BYTES:
        flush = torch.empty(512 * 2 ** 20 // 4, dtype=torch.float32, device=device)
    for t in range(1, warmup + 1):
        run(t)
    torch.cuda.synchronize()
    launch_ms, region_ms = time_launches(run, warmup + 1, steps, flush, stream)
    kernel_ms = statistics.mean(launch_ms)
    step_ms = kernel_ms if flush is not None else region_ms / steps
    peak, peak_kind = measured_peak()
    bpp = w.bytes_per_param()
    gbs = bpp * w.n / (kernel_ms / 1e3) / 1e9
    entry = {"workload": name, "mode": w.mode, "params": w.n, "tensors": len(w.sizes),
             "steps": steps, "warmup": warmup, "bytes_per_param": bpp,
             "us_per_step": step_ms * 1e3, "params_per_s": w.n / (step_ms / 1e3),
             "gb_s": gbs, "frac": gbs / peak, "peak_source": peak_kind,
             "kernel": kernel_name(w), "kernel_ms": kernel_ms,
             "kernel_ms_median": statistics.median(launch_ms), "l2": l2_policy(w, flush),
             "gpu_launches": steps * (2 if w.mode == "turbo" else 1),
             "nonfinite": int(nonfinite.item())}
    if w.mode == "turbo":
        entry["note"] = ("TurboAdam-style step (UState first moment, 1Q second moment); "
                         "the oracle baseline runs on one thread")
    if name == "single-4096":
        entry["note"] = "launch-latency bound: the fraction of peak is not meaningful here"
    entry["cpu_baseline"] = cpu_baseline(w, cpu_seconds)
    return entry


def measure_e2e(pa, w, hy, args, stream, nonfinite):
    """The step through the public API with the workload in pinned host
    memory.  Packed E4 (one tensor): pa_adamw_step_packed_e4_host, whose step
    kernel reads and writes the pinned arrays in place over the host link;
    other modes: host-to-device copies of every input, the step, device-to-host
    copies of every output, one after the other.  All of it is inside the timed
    region.  Each of the node's ranks pins its own buffers, so a rank may use at
    most 60 % of the available host memory divided by the number of ranks;
    beyond that the measurement is skipped (value null)."""
    import torch

    if w.mode == "blockwise":
        dev_in = [w.p, w.g, w.m_code, w.m_absmax, w.v_code, w.v_absmax]
        dev_out = [w.p_bf16, w.m_code, w.m_absmax, w.v_code, w.v_absmax]
    else:
        dev_in = [w.p, w.g, *w.s]
        dev_out = [w.p, *w.s]
    need = sum(t.numel() * t.element_size() for t in set(dev_in + dev_out))
    avail = host_available_bytes()
    ranks = int(os.environ.get("LOCAL_WORLD_SIZE", os.environ.get("WORLD_SIZE", "1")))
    if avail is not None and need > 0.6 * avail / max(ranks, 1):
        return {"_ms": float("nan"), "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0,
                "skipped": f"pinned host buffers of {need / 1e9:.0f} GB per rank exceed 60% of the "
                           f"{avail / 1e9:.0f} GB available shared by {ranks} rank(s)"}
    host = {id(t): torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_in + dev_out}
    for t in dev_in + dev_out:
        host[id(t)].copy_(t)
    h2d = sum(t.numel() * t.element_size() for t in dev_in)
    d2h = sum(t.numel() * t.element_size() for t in dev_out)
    if w.mode == "e4" and len(w.sizes) == 1 and not w.grad_bf16:
        ws = torch.empty(3 * 12 * (1 << 26), dtype=torch.uint8, device=w.p.device)
        hp, hg, hs = host[id(w.p)], host[id(w.g)], host[id(w.s[0])]
        api = ("pa_adamw_step_packed_e4_host (pinned host tensors, read and written in place over "
               "the host link by the step kernel; its 2.4 GB workspace is not used then)")

        def one(t):
            pa.pa_adamw_step_packed_e4_host(hp, hg, hs, ws, t, nonfinite=nonfinite, **hy)
    else:
        run = step_fn(pa, w, hy, nonfinite)
        api = "pa_adamw_step_* with pinned-host copies before and after"

        def one(t):
            for d in dev_in:
                d.copy_(host[id(d)], non_blocking=True)
            run(t)
            for d in dev_out:
                host[id(d)].copy_(d, non_blocking=True)

    one(10_000)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for k in range(args.e2e_steps):
        one(10_001 + k)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.e2e_steps
    del host
    return {"_ms": ms, "unit": "params/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "api": api}


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch

    mode = {"blockwise-1e9": "blockwise", "turbo-124m": "turbo"}.get(args.workload, args.mode)
    cores = host_cores() if mode != "turbo" else 1
    total = tensor_sizes(args.workload)[0] if args.workload in ("flat-7e9", "blockwise-1e9") \
        else wl.WORKLOADS[args.workload]["n"]
    g_fill = wl.fill_turbo_grads_ if mode == "turbo" else None
    budget = 150.0  # seconds for the whole run
    per_step = min(10.0, budget / max(1, args.steps + args.warmup))
    s = sample_size(mode, per_step, cores, total)
    p = wl.fill_normal_(torch.empty(s, dtype=torch.float32), 0.02, 1234)
    g = g_fill(torch.empty(s), 1234) if g_fill else sample_gradient(args.workload, s, 1234)
    p, g = p.numpy(), g.numpy()
    import oracle

    hy = wl.HYPER
    if mode == "blockwise":
        q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
        nb = wl.blocks(s)
        st = [np.full(s, wl.nearest_zero_code(q1), np.uint8), np.zeros(nb, np.float32),
              np.full(s, wl.nearest_zero_code(q2), np.uint8), np.zeros(nb, np.float32)]
    elif mode == "fp32":
        st = [np.zeros(s, np.float32), np.zeros(s, np.float32)]
    elif mode == "turbo":
        st = [oracle.turbo_zero_state(s)]
    else:
        st = [np.zeros(s, np.uint32)]

    def one(t):
        nonlocal p, st
        if mode == "turbo":
            p, ts, _ = oracle.turbo_step(p, g, st[0], t, **hy)
            ts["uscal"] = oracle.turbo_finalize(ts["uscal"], s)
            st = [ts]
        elif mode == "blockwise":
            _, mc, ma, vc, va, _ = oracle.step_blockwise8(p, g, st[0], st[1], st[2], st[3], q1, q2,
                                                          t, threads=cores, **hy)
            st = [mc, ma, vc, va]
        elif mode == "fp32":
            p, st[0], st[1], _ = oracle.step_fp32(p, g, st[0], st[1], t, threads=cores, **hy)
        else:
            p, st[0], _ = oracle.step_packed(p, g, st[0], t, mode=mode, threads=cores, **hy)

    for t in range(1, args.warmup + 1):
        one(t)
    t0 = time.perf_counter()
    for k in range(args.steps):
        one(args.warmup + 1 + k)
    el = time.perf_counter() - t0
    value = s * args.steps / el
    sample = (f"first {s} parameters of the {args.workload} workload per step "
              f"(of {total}), {cores} host threads")
    line = {
        "impl": "reference",
        "metric": "packed-E4 AdamW step: params/s and HBM GB/s as % of GB300 peak, 1 GPU"
                  if mode == "e4" else f"{mode} AdamW step: params/s and HBM GB/s",
        "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "mode": mode, "params_per_step": s,
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.params is not None:
        if args.workload not in ("flat-7e9", "blockwise-1e9", "turbo-124m"):
            raise SystemExit("--params applies to the one-tensor workloads only")
        PARAMS_OVERRIDE[args.workload] = args.params
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
