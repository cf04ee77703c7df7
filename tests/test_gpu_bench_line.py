"""bench.py's own arm on the GPU: one JSON line with every key the contract
asks for, consistent with itself (a short run of the 32-request workload)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_our_arm_prints_a_complete_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "b32_c32k_s4096",
                        "--steps", "5", "--warmup", "3", "--no-sweep", "--no-ce", "--no-cpu-baseline",
                        "--configs", "tiny_b1_c8k"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
                "e2e", "gpu_launches", "clocks", "step_ms_quantiles"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] == 3
    assert line["unit"] == "resolves/s" and line["value"] > 0
    # value is B * layers * steps over the summed step time
    assert abs(line["value"] - 32 / (line["ms_per_step"] / 1e3)) / line["value"] < 1e-6
    roof = line["roofline"]
    assert roof["bound"] == "h2d" and roof["unit"] == "GB/s" and 0 < roof["frac"] < 1.5
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert line["gpu_launches"] == 5  # one fused launch per step at 32 requests
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 32 * 2048 * 4
    assert line["config"]["workload"].startswith("b32_c32k_s4096")
    # the same config keys as the reference arm, the pages' figures as context
    assert set(line["config"]) == {"workload", "prime_steps_untimed", "l2", "parallelism"}
    assert len(line["context"]["figures"]) == 2
    # the other workload, measured by the same passes
    tiny = line["configs"]["tiny_b1_c8k"]
    assert tiny["value"] > 0 and tiny["steps"] == 5 and tiny["roofline"]["frac"] > 0
    assert tiny["step_roofline"]["frac"] > 0 and tiny["e2e"]["value"] > 0
    assert abs(tiny["value"] - 1 / (tiny["ms_per_step"] / 1e3)) / tiny["value"] < 1e-6
