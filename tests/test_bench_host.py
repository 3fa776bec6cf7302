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


def test_parse_clocks(tmp_path):
    """Median clock under load, the maximum, and every throttle reason seen
    Active (rows that are not samples are skipped)."""
    p = tmp_path / "clocks.csv"
    p.write_text("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                 "0, 2070, 2070, 1100.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "garbage line\n"
                 "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.parse_clocks(str(p))
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
