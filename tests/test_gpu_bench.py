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
    assert e2e["pipelined"] is True and e2e["serial"]["unit"] == d["unit"] and e2e["serial"]["value"] > 0
    assert e2e["same_loop_without_copies_ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_bench_line_plain_decode():
    """Small workload: the plain decode with one partition per sequence (no merge kernel),
    plus the read-only ceiling pass (one launch per timed step)."""
    d = run_bench("--config", "tiny", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1", "--no-extra-configs")
    check_contract(d, 5, 3)
    # fused step (1) + decode pass (append + decode: 2) + two-call pass (2) + serial e2e (the fused
    # step and its two staging copies: 3) + pipelined e2e with and without its copies (the fused
    # step; the copies are copy-engine transfers: 1 + 1), per step; the read pass
    assert d["gpu_launches"] == (1 + 2 + 2 + 3 + 2) * 5 + 5
    assert d["two_call_step_us"] > 0 and "paged_append_decode" in d["step_call"]
    rc = d["read_ceiling"]
    assert rc["us"] > 0 and rc["gbs"] > 0 and abs(rc["frac"] - rc["gbs"] / d["roofline"]["peak"]) < 1e-3
    assert d["configs"] == {} and d["seq_steps_per_s"] > 0


def test_bench_line_cascade():
    """Shared-prefix workload through the cascade call: append, prefix pass, decode and the
    merge kernel (bf16 pools merge the prefix records there)."""
    d = run_bench("--config", "prefix_shared", "--cascade", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1",
                  "--no-extra-configs")
    check_contract(d, 3, 3)
    # append, prefix pass, decode, merge: five timed passes (step, decode, serial e2e, pipelined
    # e2e with and without its copies), the serial e2e one with two staging copies
    assert d["gpu_launches"] == 4 * 3 * 5 + 2 * 3
    assert "cascade_prefix_tc_kernel" in d["roofline"]["kernel"]


def test_bench_line_times_the_other_target_workloads():
    """The default line also times the 70B-shaped long-context decode and both cascades under
    the same protocol, each with its own roofline fraction and sequence-steps per second."""
    d = run_bench("--config", "tiny", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1", "--no-e2e")
    assert set(d["configs"]) == {"long_context_70b", "prefix_shared_cascade", "fp8_fork_cascade"}
    for name, e in d["configs"].items():
        for k in ("decode_us", "decode_us_p10_p50_p90", "unique_kv_gbs", "roofline_frac", "frac_of_8tbs",
                  "seq_steps_per_s", "step_us", "config", "clocks"):
            assert k in e, (name, k)
        assert e["decode_us"] > 0 and 0 < e["roofline_frac"] < 2 and e["seq_steps_per_s"] > 0
    assert "read_ceiling" in d["configs"]["long_context_70b"]
    assert d["configs"]["fp8_fork_cascade"]["config"]["kv_dtype"] == "e4m3"


def test_reference_arm_prints_the_same_config():
    ours = run_bench("--config", "tiny", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1", "--no-extra-configs",
                     "--no-e2e", "--no-read-ceiling")
    ref = run_bench("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "0", "--cpu-seconds", "1")
    assert ref["impl"] == "reference" and ref["config"] == ours["config"]
    assert ref["metric"] == ours["metric"] and ref["unit"] == ours["unit"]
