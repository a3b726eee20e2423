"""bench.py's reference arm (no GPU): `--impl reference` times the fp64
oracle on the host cores and prints the same JSON line as the GPU arm, with
`"impl": "reference"`; under torchrun only rank 0 runs it and the other
ranks exit 0 without output."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "toy_f32", "--steps", "3", "--warmup", "1"],
                          capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_line():
    r = _run(0, 1)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == "moe_layer_tokens_per_s" and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["value"] > 0 and (j["steps"], j["warmup"], j["n_gpus"]) == (3, 1, 1)
    assert j["config"]["workload"] == "toy_f32_moe_layer"
    assert j["dtype"] == "f64" and j["data"] == "synthetic"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"] and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(1, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
