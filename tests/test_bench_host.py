"""Host-side pieces of bench.py that need no GPU."""
import os
import sys

import pytest

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


def test_timeline_split_adds_up_to_the_span():
    """Every instant goes to the running CTA that finishes next (a CTA that
    runs inside another's lifetime takes its own stretch), a gap with no CTA
    is idle, and the charges plus idle equal the span."""
    import numpy as np
    from lookahead_decoding_gb300._lib import timeline_split
    # start, end, kernel id, CTA, CTAs  (ns; ids 13 pack, 0 tensor-core GEMM, 5 RMSNorm, 2 fused attention)
    rec = np.array([[0, 100, 13, 0, 1],
                    [90, 300, 0, 0, 152],
                    [250, 280, 5, 0, 64],
                    [295, 400, 2, 0, 128],
                    [450, 470, 0, 1, 152]], dtype=np.int64)
    s = timeline_split(rec)
    assert s["ns"] == {"gemm": 190, "attention": 100, "rowwise": 30, "state": 100, "chain": 0}
    assert s["by_kernel_ns"] == {"k_gemm_tc": 190, "k_attn_fused": 100, "k_rmsnorm": 30, "k_pack": 100}
    assert s["ctas"] == {"k_gemm_tc": 2, "k_attn_fused": 1, "k_rmsnorm": 1, "k_pack": 1}
    assert s["idle_ns"] == 50 and s["span_ns"] == 470
    assert sum(s["ns"].values()) + s["idle_ns"] == s["span_ns"]
    assert timeline_split(rec[:0])["span_ns"] == 0
    # random intervals: the identity holds whatever the overlap
    rng = np.random.default_rng(1)
    st = np.sort(rng.integers(0, 10_000, 300))
    r = np.stack([st, st + rng.integers(0, 500, 300), rng.integers(0, 22, 300), np.zeros(300, int),
                  np.ones(300, int)], axis=1).astype(np.int64)
    q = timeline_split(r)
    assert sum(q["ns"].values()) + q["idle_ns"] == q["span_ns"] == int(r[:, 1].max() - r[0, 0])


def test_split_difference_is_per_call():
    """The batched line's per-call split: the longer timeline's charges minus
    the shorter one's, per kind and per kernel, over the calls between them
    (a kind absent from the shorter run counts from zero; a kernel whose
    charge does not grow, like a shared prefill's, is left out)."""
    long = {"ns": {"gemm": 5_000_000, "attention": 1_000_000, "rowwise": 0, "state": 300_000},
            "by_kernel_ns": {"k_gemm_tc": 5_000_000, "k_attn_fused": 1_000_000, "k_pack": 300_000,
                             "k_prefill_rows": 999}}
    short = {"ns": {"gemm": 1_000_000, "attention": 200_000, "rowwise": 0},
             "by_kernel_ns": {"k_gemm_tc": 1_000_000, "k_attn_fused": 200_000, "k_prefill_rows": 1000}}
    d = bench.split_difference(long, short, 4)
    assert d["ms"] == pytest.approx({"gemm": 1.0, "attention": 0.2, "state": 0.075}, rel=1e-12)
    assert d["by_kernel_ms"] == pytest.approx({"k_gemm_tc": 1.0, "k_attn_fused": 0.2, "k_pack": 0.075}, rel=1e-12)


def test_workloads_are_complete():
    """Every single-request workload names its model shape, prompt kind and
    knobs; the sampled one runs 16 prompts at temperature 0.8, top-p 0.9."""
    import synth
    for name, wl in bench.WORKLOADS.items():
        for key in ("desc", "model", "prompt", "prompt_len", "max_new", "seed", "knobs", "options", "cfg"):
            assert key in wl, (name, key)
        assert hasattr(synth, wl["cfg"]) and wl["prompt"] in ("markov", "code")
    s = bench.WORKLOADS["sampled-7b"]
    assert s["n_prompts"] == 16 and s["sampling"] == (0.8, 0.9) and s["prompt_len"] == 256
