"""bench.py's output contract: one JSON line with the keys and types the
benchmark driver reads. The reference arm (the CPU oracle) runs anywhere; the
CUDA arm needs a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BASE_KEYS = {"metric": str, "value": (int, float), "unit": str, "n_gpus": int, "steps": int, "warmup": int,
             "ms_per_step": (int, float), "higher_is_better": bool, "scaling": str, "dtype": str, "data": str,
             "config": dict}


def run_bench(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def check_base(d):
    for k, t in BASE_KEYS.items():
        assert k in d and isinstance(d[k], t), (k, d.get(k))
    assert "vs_baseline" in d and d["vs_baseline"] is None
    assert "workload" in d["config"]
    assert d["value"] > 0 and d["ms_per_step"] > 0
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "2", "--warmup", "0", "--workload", "s64_b2_h384_bf16")
    check_base(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_cuda_arm_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = run_bench("--steps", "5", "--warmup", "3", "--workload", "s4096_b8_h2048_bf16", "--no-extras")
    check_base(d)
    rf = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert d["gpu_launches"] == 2 * d["steps"]
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and "reasons" in c
    assert d["config"]["l2"].startswith("flushed")   # a 403 MB call is flushed by default
