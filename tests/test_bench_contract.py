"""bench.py's contract on the CPU: the reference arm (the fp64 oracle, timed on the host)
prints one complete JSON line, and the GPU arm fails loudly where there is no GPU instead
of falling back to anything."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_complete_line():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "0",
                  "--workload", "bf16_b2h8n1024d64")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("attention fwd TFLOPS")
    assert d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1
    assert d["warmup"] >= 3                      # at least three warm-up steps, always
    assert d["config"]["workload"] == "bf16_b2h8n1024d64"
    assert "flushed before every timed call" in d["config"]["l2"]   # 6 MiB sets fit in L2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_fails_without_a_gpu():
    r = run_bench("--steps", "1", "--warmup", "3", "--cpu-budget", "0", timeout=120)
    assert r.returncode != 0
    assert not r.stdout.strip()                  # no bench line without the CUDA path


def test_l2_handling_follows_input_set_size():
    """Input sets larger than L2 alternate without a flush; smaller ones are flushed before
    every timed call (the timing rule for inputs that fit in L2)."""
    sys.path.insert(0, ROOT)
    import bench
    from attention_forward_04_gb300.inputs import WORKLOADS
    head = WORKLOADS["bf16_b4h16n4096d128"]
    assert bench.input_set_bytes(head) == 3 * 4 * 16 * 4096 * 128 * 2
    assert bench.input_set_bytes(head, "bwd") == 5 * 4 * 16 * 4096 * 128 * 2 + 4 * 4 * 16 * 4096
    assert bench.input_set_bytes(WORKLOADS["fp8_b4h16n4096d128"]) == 3 * 4 * 16 * 4096 * 128
    assert bench.input_set_bytes(WORKLOADS["fp32_b1h1n256d64"]) == 3 * 256 * 64 * 4
    assert "no flush" in bench.l2_note(bench.input_set_bytes(head))
    for name in ("bf16_b2h8n1024d64", "fp32_b1h1n256d64", "fp8_b4h16n4096d128"):
        assert "flushed before every timed call" in bench.l2_note(bench.input_set_bytes(WORKLOADS[name]))
    assert bench.flush_buffer(torch, "cpu", bench.input_set_bytes(head)) is None
    assert bench.L2_BYTES < bench.FLUSH_BYTES


def test_backward_launch_count_per_call():
    # gpu_launches of a backward line counts the kernels of every call
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(bench)
    finally:
        sys.argv = argv
    from attention_forward_04_gb300.inputs import WORKLOADS
    assert bench.bwd_launches_per_call(WORKLOADS["bf16_b4h16n4096d128"]) == 2
    assert bench.bwd_launches_per_call(WORKLOADS["bf16_b4h8n4096d256"]) == 3
    assert bench.bwd_launches_per_call(WORKLOADS["fp32_b1h1n256d64"]) == 2
