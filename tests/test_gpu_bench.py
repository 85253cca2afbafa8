"""The benchmark's JSON line on a GPU: one line with the keys and units its readers use, the
roofline of the decode kernel, the end-to-end figure, the oracle baseline, the clocks and
a launch count that matches the kernels of a step (append, [prefix pass], decode, [merge])
times the timed passes (device step, decode alone, end to end) times the steps."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def check_contract(d, steps, warmup):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "cpu_baseline", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup and d["warmup"] >= 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert "workload" in d["config"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0 and rf["achieved"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and 0 < e2e["value"] and e2e["h2d_bytes_per_step"] > 0
    assert e2e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_bench_line_plain_decode():
    """Small workload: the plain decode with one partition per sequence (no merge kernel)."""
    d = run_bench("--config", "tiny", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1")
    check_contract(d, 5, 3)
    assert d["gpu_launches"] == 2 * 3 * 5  # append + decode, three timed passes


def test_bench_line_cascade():
    """Shared-prefix workload through the cascade call: append, prefix pass, decode and the
    merge kernel (bf16 pools merge the prefix records there)."""
    d = run_bench("--config", "prefix_shared", "--cascade", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1")
    check_contract(d, 3, 3)
    assert d["gpu_launches"] == 4 * 3 * 3
    assert "cascade_prefix_tc_kernel" in d["roofline"]["kernel"]
