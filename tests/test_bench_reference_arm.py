"""bench.py's reference arm on CPU: the fp64 oracle on the host's threads,
one JSON line with the fields the reference arm must carry."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] >= 3 and line["higher_is_better"] is True
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["cores"] >= 1
    assert cpu["cpu_model"] and "host threads" in cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
