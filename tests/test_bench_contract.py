"""bench.py's command line on the CPU: the reference arm (the oracle, timed on the host
cores) prints one JSON line with the contract's keys on the same metric as the GPU arm,
and the GPU arm refuses to run without a GPU instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--workload", "tiny_f32", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    sys.path.insert(0, ROOT)
    import bench
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["impl"] == "reference" and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["vs_baseline"] is None
    assert line["data"] == "synthetic" and line["scaling"] in ("weak", "strong")
    assert line["config"]["workload"] == "tiny_f32"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_gpu_arm_refuses_without_a_gpu():
    if torch.cuda.is_available():
        return
    r = _bench("--workload", "tiny_f32", "--steps", "3", "--warmup", "3")
    assert r.returncode != 0
    assert not r.stdout.strip(), "the GPU arm printed a result without a GPU"
