"""GPU: bench.py prints one JSON line with every key its contract names, for the
device arm (small decode batch) and for the reference arm (the oracle)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_device_arm_json_contract():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--steps", "2", "--warmup", "3", "--decode-batch", "2", "--configs", "wide"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "bf16"
    assert "workload" in d["config"]
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] in ("hbm", "tensor") and r["frac"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in d["e2e"], key
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in cb, key
    assert cb["kind"] == "oracle" and cb["cores"] >= 1
    # prefill (plus the key-rotation pass where it runs) + decode split + combine per step
    pre = 2 if d["roofline_prefill"]["kernel"].startswith("rope_keys_kernel") else 1
    assert d["gpu_launches"] == (pre + 2) * d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    c = d["configs"]["wide"]
    for key in ("workload", "ms_per_call", "value", "unit", "roofline"):
        assert key in c, key
    assert c["roofline"]["bound"] == "tensor" and c["roofline"]["frac"] > 0
    assert abs(c["roofline"]["frac"] - c["roofline"]["achieved"] / c["roofline"]["peak"]) < 1e-9


def test_reference_arm_json_contract():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "config", "cpu_baseline",
                "e2e"):
        assert key in d, key
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"
