"""The benchmark's command line on the CPU: the reference arm (the float64
oracle timed on host cores) prints one JSON line with the fields of the GPU
arm's line, and the GPU arm fails loudly instead of falling back to the CPU
when there is no CUDA device."""

import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                          text=True, timeout=600, env=env)


def test_reference_arm_prints_one_json_line():
    p = _run(["--impl", "reference", "--steps", "1", "--warmup", "0", "--cpu-tokens", "256"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1
    assert d["config"]["workload"] == "bf16_gqa_s64k_h32kv8_d128_c8_zigzag"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a CUDA device")
def test_gpu_arm_fails_without_cuda():
    p = _run(["--steps", "1", "--warmup", "0", "--no-cpu-baseline", "--no-ulysses", "--no-linear"])
    assert p.returncode != 0
    assert not any(l.startswith("{") for l in p.stdout.splitlines())


def test_reference_arm_takes_the_overrides():
    p = _run(["--impl", "reference", "--steps", "1", "--warmup", "0", "--cpu-tokens", "256", "--cp-size", "4",
              "--heads", "16:4", "--seq-len", "32768", "--seed", "3"])
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads([l for l in p.stdout.splitlines() if l.startswith("{")][0])
    c = d["config"]
    assert (c["total_tokens"], c["hq"], c["hkv"], c["cp_size"]) == (32768, 16, 4, 4)
    assert c["workload"].startswith("bf16_gqa_s64k_h32kv8_d128_c8_zigzag[")


def test_bad_override_is_refused():
    p = _run(["--impl", "reference", "--steps", "1", "--warmup", "0", "--heads", "6:4"])
    assert p.returncode != 0
    p = _run(["--impl", "reference", "--steps", "1", "--warmup", "0", "--seq-len", "-5"])
    assert p.returncode != 0


def test_varlen_pack_takes_a_token_count():
    p = _run(["--impl", "reference", "--steps", "1", "--warmup", "0", "--cpu-tokens", "256", "--workload",
              "bf16_varlen_t128k_h16kv4_d128_c16_zigzag", "--seq-len", "32768"])
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads([l for l in p.stdout.splitlines() if l.startswith("{")][0])
    assert d["config"]["total_tokens"] == 32768
    assert d["config"]["workload"] == "bf16_varlen_t128k_h16kv4_d128_c16_zigzag[total_tokens=32768]"
