"""The benchmark's JSON line on the GPU: one short run of bench.py on the 8k-prefix workload,
checked for every key the result line carries (metric, throughput, roofline with the DRAM
traffic of the committed ncu summary, end-to-end figures with their copy sizes, kernel
launches, clock samples)."""
import json
import os
import subprocess
import sys

import pytest

from parity_util import require_cuda

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    require_cuda()
    r = subprocess.run([sys.executable, "bench.py", "--config", "c2", "--also=", "--steps", "5", "--warmup", "3",
                        "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("c2")
    roof = line["roofline"]
    assert roof["bound"] in ("tensor", "hbm") and 0 < roof["frac"] < 1.5
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert roof["traffic"] is not None and roof["traffic"] > 0  # the committed summary matches the source
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["pipelined"]["value"] > 0
    assert line["gpu_launches"] == 2 * line["steps"]           # prefix pass + tail/merge per step
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
