"""bench.py prints one JSON line carrying the measurement contract's keys
(the 8k-token workload as the headline and the tiny one as a per-config
record, so the run takes seconds)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    cmd = [sys.executable, "bench.py", "--workload", "8k", "--steps", "3", "--warmup", "3",
           "--cpu-rows", "4", "--configs", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["scaling"] == "weak" and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("8k")
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and rf["unit"] in ("GB/s", "TFLOP/s")
    assert rf["achieved"] > 0 and rf["peak"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert "traffic" in rf
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    # e2e returns the step's results, not only the loss
    assert e2e["d2h_bytes_per_step"] > e2e["h2d_bytes_per_step"] / 2
    pc = d["per_config"]
    assert set(pc) == {"8k", "tiny"}, set(pc)
    for name, rec in pc.items():
        assert rec["ms_per_step"] > 0 and rec["tflops"] > 0 and rec["tokens_per_s"] > 0, name
        assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] > 0, name
        assert "dense_sdpa" in rec, name
    assert pc["tiny"]["cpu_baseline"]["sample"].startswith("every row")
    assert set(pc["tiny"]["kernels_ms"]) == {"k_select", "k_fwd", "k_bwd"}
