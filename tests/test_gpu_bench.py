"""bench.py's output contract: one JSON line with the keys the harness reads,
for the native arm and for the reference (oracle) arm."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args) -> dict:
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_native_line_has_the_contract_keys():
    d = _run("--steps", "5", "--warmup", "3", "--seeds", "2", "--cpu-seconds", "2")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert "workload" in d["config"]
    assert d["config"]["name"] == "large_bf16"  # the largest single-GPU configuration
    for key in ("large_fp8", "skewed_seeds", "verify"):  # the target's evidence, in the same line
        assert key in d, key
    for name in ("skewed_mtp3", "rows_fp8_t3", "mtp_verify"):  # multi-token verify rows
        v = d["verify"][name]
        assert v["us_per_decode_call"] > 0 and 0 < v["call_frac_of_measured"]
    sk = d["skewed_seeds"]
    assert sk["seeds"] == 2 and len(sk["per_seed"]) == 2
    for k in ("call_frac_of_measured", "split_frac_of_measured",
              "uniform_over_proportional_call"):
        assert sk[k]["median"] > 0 and sk[k]["p10"] > 0
    assert d["large_fp8"]["us_per_decode_call"] > 0
    assert d["e2e_kv_resident"]["h2d_bytes_per_step"] < d["e2e"]["h2d_bytes_per_step"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert 0 < rf["achieved"] and 0 < rf["peak"]
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    # planner and split kernel per step, and the merge kernel unless it is fused
    assert d["gpu_launches"] in (2 * 5, 3 * 5)
    assert d["clocks"]["sm_max_mhz"] > 0


def test_reference_line_has_the_contract_keys():
    d = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
