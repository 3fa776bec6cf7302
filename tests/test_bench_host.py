"""Host-side pieces of bench.py that need no GPU."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
import synth  # noqa: E402


def test_cpu_oracle_sample_is_bounded_and_reports_its_sample():
    cfg = synth.TINY
    w = synth.llama_weights(cfg, 0)
    s = bench.cpu_oracle_sample(cfg, w, min_s=0.05, max_calls=3, prompt_len=8)
    assert s["kind"] == "oracle" and s["unit"] == "tokens/s" and s["value"] > 0
    assert s["cores"] >= 1
    assert "packed calls" in s["sample"]
