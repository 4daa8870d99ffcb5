"""bench.py --impl reference (the CPU oracle arm) prints one JSON line with the
contract's keys; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"]
    # the oracle's step time is a scaled-up sample, and says so
    assert d["extrapolated"] is True and d["sample_seconds_per_step"] > 0
    # the same config keys as the device arm's line
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    ns = argparse.Namespace(gpus=1, path="dual", sr="philox16", graph=1)
    assert d["config"] == bench.main_config(ns)
    assert d["cpu_baseline"]["quantize_gbs"] > 0 and d["cpu_baseline"]["gemm_tflops"] > 0


def test_input_digests_are_stable():
    """The bench's input digests depend only on the seeded generators."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import synth
    a = bench.input_digests(x=synth.normal_bf16((64, 128), 5, 1.0, 0.0005, 100.0))
    b = bench.input_digests(x=synth.normal_bf16((64, 128), 5, 1.0, 0.0005, 100.0))
    c = bench.input_digests(x=synth.normal_bf16((64, 128), 6, 1.0, 0.0005, 100.0))
    assert a == b and a != c and len(a["x"]) == 64
    assert bench.input_digests(z=np.zeros(4, np.uint16))["z"] == \
        "af5570f5a1810b7af78caf4bc70a660f0df51e42baf91d4de5b2328de0e83dfc"
