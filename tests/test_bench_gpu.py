"""bench.py end to end on the GPU: one JSON line per run with the contract's
keys, for the L2-flush and rotating-input modes, a dense workload with its
end-to-end leg and the batched workload (one grouped launch per step)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
        "cpu_baseline", "e2e", "gpu_launches", "clocks")


def _bench(*args):
    r = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3", *args],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    for k in KEYS:
        assert k in line, k
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["n_gpus"] == 1
    assert line["roofline"]["frac"] > 0 and line["roofline"]["peak"] > 0
    assert line["gpu_launches"] >= 3
    return line


@pytest.mark.parametrize("flush", ["write+read", "rotate"])
def test_bench_line_dense_with_end_to_end(flush):
    line = _bench("--workload", "fp16_1024_uniform", "--flush", flush, "--cpu-budget", "0.5")
    assert line["config"]["workload"] == "fp16_1024_uniform"
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["ms_per_call_median"] <= e2e["ms_per_call_max"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] > 0
    assert ("copies of the inputs" in line["config"]["l2"]) == (flush == "rotate")


def test_bench_line_batched():
    line = _bench("--workload", "fp16_batched_16x1024x1024x1024", "--no-cpu-baseline",
                  "--no-e2e")
    assert line["config"]["kernel"]["launches"] == 1
    assert line["e2e"] is None and line["cpu_baseline"] is None
