"""The benchmark's reference arm on CPU: the oracle on the host cores, with the per-step token
sample shrunk so that the whole run stays within its time bound, printing the contract's line."""
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_is_bounded_and_prints_the_contract_line():
    t0 = time.time()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "40",
                          "--warmup", "3", "--ref-total-seconds", "4"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 40 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and 1 <= cb["cores"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    n = line["config"]["tokens_per_step"]
    assert 1 <= n <= 8192 and cb["cores"] <= n
    # 43 steps of the bounded sample: the oracle work stays near the 4 s bound (input generation
    # and the calibration run come on top)
    assert line["ms_per_step"] * 43 / 1e3 < 4 * 3
    assert time.time() - t0 < 600
