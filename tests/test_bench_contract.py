"""The bench's JSON line on the host: the reference arm (the fp64 oracle on the host cores) on the
256-token workload, and the argument checks that need no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=120):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    r = _bench("--impl", "reference", "--workload", "tiny_full_f32_B1_H4_S256_d64", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == "attention fwd useful TFLOP/s and % of GB300 dense BF16 tensor peak"
    assert line["unit"] == "TFLOP/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 3
    assert line["config"]["workload"] == "tiny_full_f32_B1_H4_S256_d64"
    assert line["data"] == "synthetic"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_rejected():
    r = _bench("--impl", "reference", "--workload", "tiny_full_f32_B1_H4_S256_d64", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0
    assert "--warmup" in r.stderr


def test_bias_matrix_with_backward_is_rejected():
    r = _bench("--bias", "--backward")
    assert r.returncode != 0
    assert "--bias" in r.stderr
