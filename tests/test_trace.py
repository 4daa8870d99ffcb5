"""NVFP4_TRACE=1 logs each binding call (name, argument shapes, time) to
stderr; checked on host-only calls, no GPU needed."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_value):
    env = dict(os.environ, NVFP4_TRACE=env_value, PYTHONPATH=ROOT)
    code = ("import nvfp4_block_scaled_29_b300 as nv; "
            "assert nv.nvfp4_scale_bytes(256, 64) == 1024; "
            "assert nv.nvfp4_rht_mask_from_seed(7) == nv.nvfp4_rht_mask_from_seed(7)")
    return subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)


def test_trace_logs_calls():
    r = _run("1")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stderr.splitlines() if l.startswith("[nvfp4]")]
    assert any(l.startswith("[nvfp4] nvfp4_scale_bytes(256, 64)") and l.endswith("(enqueue)") for l in lines), lines
    assert sum("nvfp4_rht_mask_from_seed(7)" in l for l in lines) == 2


def test_no_trace_by_default():
    r = _run("")
    assert r.returncode == 0, r.stderr
    assert "[nvfp4]" not in r.stderr
