"""Host-side logic of bench.py, on the CPU: the workload shapes it steps and
the rule that reports ncu traffic only for the kernel code it was taken on."""
import hashlib
import importlib.util
import json
import os
import shutil

import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = ("packedadam.cu", "codecs.cuh", "blockwise.cuh", "pipeline.cuh", "f32x2.cuh",
           "turbo.cuh", "exact.cuh")


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_workload_shapes(bench):
    """The configurations' tensor lists: 52 tensors of 9,677,312 parameters
    (biases folded into their weights), GPT-2 small's 148 tensors of
    124,439,808, one tensor each for the flat and blockwise workloads."""
    g52 = bench.tensor_sizes("gpt-52")
    assert len(g52) == 52 and sum(g52) == 9_677_312
    assert g52[:2] == [3_096_576, 262_144]
    assert g52[2:8] == [197_376, 65_792, 263_168, 262_400, 512, 512]
    g2 = bench.tensor_sizes("gpt2-148")
    assert len(g2) == 148 and sum(g2) == 124_439_808
    assert bench.tensor_sizes("flat-7e9") == [7_000_000_000]
    assert bench.tensor_sizes("single-4096") == [4096]
    n = bench.tensor_sizes("blockwise-1e9")[0]
    assert wl.blocks(n) == 488_282 and n - (wl.blocks(n) - 1) * 2048 == 512


def _tree(tmp_path):
    src = os.path.join(ROOT, "adamw_update_gb300", "csrc")
    dst = tmp_path / "adamw_update_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    (tmp_path / "profiles").mkdir()
    return dst


def test_traffic_is_reported_only_for_the_captured_code(bench, tmp_path, monkeypatch):
    dst = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_per_param("e4") is None  # no record
    digest = hashlib.sha256(bench.kernel_code_digest_input().encode()).hexdigest()
    record = {"e4": {"source_sha256": digest, "dram_bytes_per_param": 19.78}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(record))
    assert bench.traffic_per_param("e4") == pytest.approx(19.78)
    assert bench.traffic_per_param("fp32") is None  # no capture of that mode
    cu = dst / "pipeline.cuh"
    text = cu.read_text()
    cu.write_text(text + "\n// a comment added after the capture\n\n")
    assert bench.traffic_per_param("e4") == pytest.approx(19.78)  # comments do not count
    cu.write_text(text.replace("2000000000ull", "1000000000ull", 1))
    assert bench.traffic_per_param("e4") is None  # the code changed


def test_committed_traffic_record_is_sane():
    """Whatever code it was taken on, the committed record's traffic is close
    to the algorithmic bytes of each mode (no re-reads)."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    algorithmic = {"e4": 20.0, "fp16": 20.0, "fp32": 28.0, "blockwise": 14.0 + 16 / 2048}
    for mode, b in algorithmic.items():
        got = rec[mode]["dram_bytes_per_param"]
        assert 0.95 * b <= got <= 1.02 * b, (mode, got)
        assert os.path.exists(os.path.join(ROOT, rec[mode]["capture"]))


@pytest.mark.parametrize("mode", ["e4", "fp32", "blockwise"])
def test_cpu_baseline_times_all_cores_and_one_thread(bench, mode):
    """The oracle arm of the bench line on a small host-resident workload."""
    import numpy as np
    import torch

    class W:
        pass

    w = W()
    w.name, w.mode, w.n = "gpt-52", mode, 1 << 16
    rng = np.random.default_rng(0)
    w.p = torch.from_numpy(rng.normal(0, 0.02, w.n).astype(np.float32))
    w.g = torch.from_numpy(rng.normal(0, 1e-3, w.n).astype(np.float32))
    if mode == "blockwise":
        q1, q2 = wl.dynamic_qmap_signed(), wl.dynamic_qmap_unsigned()
        nb = wl.blocks(w.n)
        w.m_code = torch.full((w.n,), wl.nearest_zero_code(q1), dtype=torch.uint8)
        w.v_code = torch.full((w.n,), wl.nearest_zero_code(q2), dtype=torch.uint8)
        w.m_absmax = torch.zeros(nb)
        w.v_absmax = torch.zeros(nb)
        w.q1, w.q2 = torch.from_numpy(q1), torch.from_numpy(q2)
    elif mode == "fp32":
        w.s = [torch.zeros(w.n), torch.zeros(w.n)]
    else:
        w.s = [torch.zeros(w.n, dtype=torch.int32)]
    cpu = bench.cpu_baseline(w, 0.2)
    assert cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["kind"] == "oracle"
    one = cpu["single_thread"]
    assert one["value"] > 0 and "1 thread" in one["sample"]


def test_configs_cover_every_benchmark_workload(bench):
    """The `configs` object of the default bench line measures all five
    workloads: single-4096 (10 steps), gpt-52 packed E4 and FP32 (100 steps
    each), gpt2-148 packed E4 and FP16 (50 steps each), flat-7e9 (the headline
    itself) and the 8-bit blockwise mode on 1e9 parameters."""
    got = {(name, mode): steps for name, mode, steps in bench.CONFIGS}
    assert got == {("single-4096", "e4"): 10, ("gpt-52", "e4"): 100, ("gpt-52", "fp32"): 100,
                   ("gpt2-148", "e4"): 50, ("gpt2-148", "fp16"): 50, ("flat-7e9", "e4"): None,
                   ("blockwise-1e9", "blockwise"): 20, ("turbo-124m", "turbo"): 20}
    assert {name for name, _, _ in bench.CONFIGS} == set(wl.WORKLOADS)


def test_configs_only_on_the_default_headline(bench):
    """The per-configuration measurements ride only on the default bench line
    (flat-7e9, packed E4, the product library, a C-ABI call per step)."""
    import sys

    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        assert bench.want_configs(bench.parse())
        for extra in (["--no-configs"], ["--params", "1024"], ["--graph"], ["--fast"],
                      ["--grad", "bf16"], ["--workload", "gpt-52"], ["--mode", "fp32"]):
            sys.argv = ["bench.py", *extra]
            assert not bench.want_configs(bench.parse()), extra
    finally:
        sys.argv = argv
