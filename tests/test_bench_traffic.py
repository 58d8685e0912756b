"""bench.py's roofline `traffic`: the ncu DRAM bytes per launch recorded in a
profile summary, looked up under the kernel the plan picked (on CPU)."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KERNEL = {"pa_tile": "tcgen05 tile", "pa_attn": "mma.sync m16n8k16"}


def test_every_recorded_summary_is_found_under_its_kernel():
    found = 0
    for f in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        m = re.fullmatch(r"(pa_tile|pa_attn)_(.+)\.txt", f)
        if not m:
            continue
        text = open(os.path.join(ROOT, "profiles", f)).read()
        rec = re.search(r"^dram_bytes_per_launch_full_size: (\d+)$", text, re.M)
        if not rec:
            continue
        kind, workload = m.groups()
        assert bench.dominant_traffic({"kernel": KERNEL[kind]}, workload) == int(rec.group(1)), f
        other = "pa_attn" if kind == "pa_tile" else "pa_tile"
        if not os.path.exists(os.path.join(ROOT, "profiles", f"{other}_{workload}.txt")):
            assert bench.dominant_traffic({"kernel": KERNEL[other]}, workload) is None
        found += 1
    assert found >= 5


def test_hbm_bound_call_on_the_tile_kernel():
    """The MQA call is HBM-bound but runs on the tile kernel: its bytes come from
    the tile kernel's summary."""
    t = bench.dominant_traffic({"kernel": "tcgen05 tile"}, "mqa_b32_t16384")
    assert t is not None and 530e6 < t < 550e6
    assert bench.dominant_traffic({"kernel": "mma.sync m16n8k16"}, "mqa_b32_t16384") is None
