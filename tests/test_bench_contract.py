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
    # the GPU arm builds its config with the same function and arguments: identical dicts
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    import workloads as wl
    args = argparse.Namespace(alibi=False, bias=False, fp8=False)
    assert line["config"] == json.loads(json.dumps(bench.fwd_config(args, wl.TINY_FULL_F32, 1)))
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


def test_bias_matrix_with_fp8_or_alibi_is_rejected():
    for extra in (("--fp8",), ("--alibi",), ("--backward", "--alibi")):
        r = _bench("--bias", *extra)
        assert r.returncode != 0
        assert "--bias" in r.stderr


def test_reference_arm_takes_the_score_bias_of_the_command_line():
    """With --bias the oracle leg adds the same bias matrix the GPU arm sets, and both arms
    print the same config."""
    r = _bench("--impl", "reference", "--workload", "tiny_full_f32_B1_H4_S256_d64", "--steps", "1", "--warmup", "3",
               "--bias")
    assert r.returncode == 0, r.stderr
    line = json.loads([l for l in r.stdout.splitlines() if l.strip()][0])
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    import workloads as wl
    args = argparse.Namespace(alibi=False, bias=True, fp8=False)
    assert line["config"] == json.loads(json.dumps(bench.fwd_config(args, wl.TINY_FULL_F32, 1)))
    assert line["config"]["score_bias"].startswith("matrix")
    alibi, bias = bench.score_bias_host(args, wl.TINY_FULL_F32)
    assert alibi is None and bias.shape == (1, 4, 256, 256) and bias.dtype.name == "float32"


def test_clock_summary_is_time_weighted_over_the_timed_region():
    """Readings outside [start, end] are dropped (the one in force at the start is kept), each
    reading weighs the time until the next, and the NVML reason bits map to their names."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.t0, c.t1 = 100.0, 100.010
    rows = [(99.990, 1500, 0)]                                   # before the region: dropped
    rows += [(99.9995, 2070, 0)]                                 # in force at the start
    rows += [(100.000 + 0.001 * k, 1800 if k < 3 else 2070, 0x4 if k == 5 else 0) for k in range(1, 10)]
    rows += [(100.020, 900, 0x40)]                               # after the region: dropped
    out = "\n".join("%.6f %d 2070 850000 %d" % r for r in rows)
    s = c._summary_nvml(out)
    assert s["samples"] == 9
    # 2070 MHz holds for 0.001 + 0.007 s, 1800 MHz for 0.002 s: the weighted median is 2070
    assert s["sm_mhz_time_weighted_median"] == 2070 and s["sm_mhz"] == 2070
    assert s["sm_mhz_min"] == 1800 and s["reasons"] == ["sw_power_cap"]
    assert abs(s["power_w_max"] - 850.0) < 1e-9 and s["sm_max_mhz"] == 2070


def test_traffic_is_read_only_from_a_summary_of_the_current_source(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary only while the summary's source hash
    equals the hash of the kernel sources as they are; any other hash, or no summary, gives None."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sources = ["k.cu"]
    h1 = bench.kernel_hash(sources)
    (prof / "kern_w.md").write_text(f"kernel_source_hash: {h1}\ndram_bytes_per_full_launch: 123456\n")
    assert bench.ncu_traffic("w", "kern", sources) == 123456.0
    assert bench.ncu_traffic("other", "kern", sources) is None  # no summary for that workload
    src.write_text("// kernel v2\n")  # the source moved on: the counters are stale
    assert bench.kernel_hash(sources) != h1
    assert bench.ncu_traffic("w", "kern", sources) is None


def test_every_committed_summary_names_its_hash_and_bytes():
    """Each profile the bench reads traffic from carries both fields (current or marked stale)."""
    import re
    names = [n for n in os.listdir(os.path.join(ROOT, "profiles"))
             if n.startswith(("attn_fwd_tc_", "attn_bwd_", "attn_decode_"))]
    assert names
    for n in names:
        text = open(os.path.join(ROOT, "profiles", n)).read()
        assert re.search(r"kernel_source_hash:\s*[0-9a-f]{16}\b", text), n
        assert re.search(r"dram_bytes_per_full_launch:\s*[0-9]+", text), n
