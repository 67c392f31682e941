"""bench.py prints one JSON line with the keys and units its contract asks
for (a short run on the GPU)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--e2e-steps", "1",
                        "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks", "per_op"]:
        assert k in d, k
    assert d["unit"] == "GB/s" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "bf16"
    assert d["gpu_launches"] == 3 * len(d["per_op"]) == 30
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and 0 < rf["frac"] < 1.3
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0 and 0 < e["value"] < d["value"]
    assert "workload" in d["config"]
    assert d["value"] > 0 and d["value"] < 1.3 * rf["peak"]
    # each step op alone, the ops beyond the step, the sweep and the small-call cost
    assert set(d["per_op_isolated"]) == set(d["per_op"])
    assert all(0 < v["frac_measured"] < 1.3 for v in d["per_op_isolated"].values())
    assert len(d["next_per_op"]) >= 10
    sw = d["sweep"]
    cells = sw["grid"]
    assert len(cells) == 2 * 4 * 5                     # dtypes x tokens x hidden sizes
    assert all("torch_copy_reference" in c for c in cells.values())
    big = {k: v for k, v in sw["largest"]["bf16"].items() if k != "torch_copy_reference"}
    assert abs(sw["largest_bf16_min_frac_nominal_8tbs"] - min(v["frac_nominal_8tbs"] for v in big.values())) < 1e-9
    hc = d["host_call_cost"]
    for k in ("python_binding_us", "c_abi_us", "torch_add_us"):
        host_us, dev_us = hc[k]
        assert 0 < dev_us <= host_us * 1.05 + 0.5
    assert 0 < hc["cuda_graph_replay_device_us"] < hc["c_abi_us"][1] * 2
