"""bench.py's host-side pieces that need no GPU: the cpu_baseline object the
JSON line carries (all host cores, then one thread)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_cpu_baseline_contract():
    import bench
    cb = bench.cpu_baseline(0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT
    assert cb["value"] > 0 and cb["cores"] >= 1 and "MLP steps" in cb["sample"]
    one = cb["one_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == bench.UNIT
