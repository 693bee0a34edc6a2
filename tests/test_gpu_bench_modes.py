"""Every bench.py mode runs end to end on a small case and prints one JSON
line: the headline steps, the second run of the same steps with events
around the main kernel, and (fused mode) the end-to-end leg."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = ["--steps", "2", "--warmup", "3", "--no-cpu-baseline", "--no-torch-ref", "--e2e-steps", "1",
         "--vocab", "16000", "--rows", "512"]


@pytest.mark.parametrize("mode,extra", [("fused", []), ("split", []), ("vp", ["--vocab-shards", "4"]),
                                        ("weighted", []),
                                        ("linear", ["--hidden", "256", "--chunk-rows", "256"]),
                                        ("linear", ["--hidden", "256", "--chunk-rows", "256",
                                                    "--linear-gemm", "library"])])
def test_bench_mode_runs(mode, extra):
    out = subprocess.run([sys.executable, "bench.py", "--mode", mode, *SMALL, *extra], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    keys = ["metric", "value", "unit", "ms_per_step", "roofline", "clocks", "config"]
    if mode == "fused":
        keys += ["e2e", "gpu_launches", "cpu_baseline"]
    for key in keys:
        assert key in line, key
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["roofline"]["frac"] > 0
