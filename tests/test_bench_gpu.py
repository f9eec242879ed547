"""bench.py end to end on the GPU, on the small 512^3 workload: the JSON line
keeps its contract (metric, value, roofline, cpu_baseline, clocks, e2e,
gpu_launches), and --role-stats reports the kernel's per-role accounting."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_bench_line_contract_small_workload():
    d = run_bench("--workload", "gemm512_uniform", "--steps", "5", "--warmup", "3", "--e2e-steps", "2")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "clocks", "e2e",
              "gpu_launches"):
        assert k in d, k
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 5 and d["gpu_launches"] == 5
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 512 * 512 * 4
    assert "workload" in d["config"] and "plan" in d["config"]


def test_role_stats_mode():
    d = run_bench("--role-stats", "--workload", "gemm512_uniform", "--steps", "5")
    per = d["us_per_cta_and_launch"]
    assert set(per) == {"mma_wait_full", "mma_wait_acc", "mma_loop_total", "producer_wait_empty",
                        "epilogue_wait_acc", "epilogue_busy"}
    assert per["mma_loop_total"] > 0 and per["epilogue_busy"] > 0
    assert all(v >= 0 for v in per.values())
