"""The bench's reference arm (the fp64 oracle on the host cores) runs without a
GPU: its one JSON line must carry the keys of the bench contract, with the
same metric, unit and direction as the GPU arm's line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(*extra):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", *extra],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit", [("tiny_gqa_d64", "GB/s"), ("chunked_prefill_q64_d64", "TFLOP/s")])
def test_reference_line_keys(workload, unit):
    extra = ["--workload", workload] + (["--cpu-budget-s", "0.5"] if "prefill" in workload else [])
    d = _reference_line(*extra)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == unit and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["value"] > 0 and d["config"]["workload"] == workload
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and cpu["unit"] == unit
    assert cpu["sample"] and cpu["cpu_model"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
