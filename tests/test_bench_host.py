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


def test_batch_prompts_are_distinct_and_seeded():
    import bench
    a = bench.batch_prompts(32000, 4)
    assert a == bench.batch_prompts(32000, 4)
    assert len({tuple(p) for p in a}) == 4 and all(len(p) == bench.PROMPT_LEN for p in a)
